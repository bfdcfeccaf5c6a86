// block_manager.cpp -- host-side physical block manager of libpagedkv.
//
// Page "大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心
// PagedAttention 显存物理布局深度剖析", section 三 (KVBlockManager and
// PagedAttentionScheduler.append_token) and section 四.2 (reference counts
// for shared prefix blocks):
//   - allocate() hands out the lowest free id (the page keeps its free list
//     sorted and pops the front) and sets its count to 1;
//   - free() decrements a held block and returns it to the free set at 0;
//   - add_reference() increments the count of a held block;
//   - append_token opens a new block when the token count is a multiple of
//     the block size, then counts the token.
// Defragmentation (page "vLLM 中 FlashAttention 与 KVCache 交换机制深度解析":
// swap_blocks also rearranges scattered pages into a compact layout): the
// used blocks move to [0, n_used).
// Copy-on-write (section 四.2): a request that writes its next token into a
// block other requests still reference gets a private copy of that block.
// The free set is a bitmap with a "lowest possibly free word" hint, so
// allocate/free cost O(1) amortised instead of the page's list sort.
#include <stdint.h>
#include <stdlib.h>

#include <new>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> ref;       // reference count per block
    std::vector<uint64_t> free_bits;  // bit set = block free
    int free_count = 0;
    int hint = 0;  // no free block lives in a word below this index

    bool is_free(int b) const { return (free_bits[b >> 6] >> (b & 63)) & 1u; }
    void mark_free(int b) {
        free_bits[b >> 6] |= (uint64_t)1 << (b & 63);
        ++free_count;
        if ((b >> 6) < hint) hint = b >> 6;
    }
    void mark_held(int b) {
        free_bits[b >> 6] &= ~((uint64_t)1 << (b & 63));
        --free_count;
    }
    int lowest_free() {
        const int words = (int)free_bits.size();
        for (int w = hint; w < words; ++w) {
            if (free_bits[w]) {
                hint = w;
                return (w << 6) + __builtin_ctzll(free_bits[w]);
            }
        }
        hint = words;
        return -1;
    }
};

static pkv_block_manager* make_manager(int num_blocks, int block_size) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    pkv_block_manager* m = new (std::nothrow) pkv_block_manager();
    if (!m) return nullptr;
    try {
        m->num_blocks = num_blocks;
        m->block_size = block_size;
        m->ref.assign((size_t)num_blocks, 0);
        m->free_bits.assign(((size_t)num_blocks + 63) / 64, 0);
    } catch (...) {
        delete m;
        return nullptr;
    }
    return m;
}

extern "C" {

PKV_API pkv_block_manager* pkv_block_manager_create(int num_blocks, int block_size) {
    pkv_block_manager* m = make_manager(num_blocks, block_size);
    if (!m) return nullptr;
    for (int b = 0; b < num_blocks; ++b) m->mark_free(b);
    m->hint = 0;
    return m;
}

PKV_API pkv_block_manager* pkv_block_manager_create_with_free(int num_blocks, int block_size,
                                                              const int32_t* free_ids,
                                                              int n_free) {
    if (n_free < 0 || (n_free > 0 && !free_ids)) return nullptr;
    pkv_block_manager* m = make_manager(num_blocks, block_size);
    if (!m) return nullptr;
    for (int b = 0; b < num_blocks; ++b) m->ref[b] = 1;
    for (int k = 0; k < n_free; ++k) {
        const int b = free_ids[k];
        if (b < 0 || b >= num_blocks || m->is_free(b)) {
            delete m;
            return nullptr;
        }
        m->ref[b] = 0;
        m->mark_free(b);
    }
    m->hint = 0;
    return m;
}

PKV_API void pkv_block_manager_destroy(pkv_block_manager* mgr) { delete mgr; }

PKV_API pkv_status pkv_block_allocate(pkv_block_manager* mgr, int32_t* block_id) {
    if (!mgr || !block_id) return PKV_ERR_INVALID;
    const int b = mgr->lowest_free();
    if (b < 0) {
        *block_id = -1;
        return PKV_ERR_NO_BLOCKS;
    }
    mgr->mark_held(b);
    mgr->ref[b] = 1;
    *block_id = b;
    return PKV_OK;
}

PKV_API pkv_status pkv_block_free(pkv_block_manager* mgr, int32_t block_id) {
    if (!mgr || block_id < 0 || block_id >= mgr->num_blocks) return PKV_ERR_INVALID;
    if (mgr->ref[block_id] > 0) {
        if (--mgr->ref[block_id] == 0) mgr->mark_free(block_id);
    }
    return PKV_OK;
}

PKV_API pkv_status pkv_block_add_reference(pkv_block_manager* mgr, int32_t block_id) {
    if (!mgr || block_id < 0 || block_id >= mgr->num_blocks) return PKV_ERR_INVALID;
    if (mgr->ref[block_id] == 0) return PKV_ERR_INVALID;
    ++mgr->ref[block_id];
    return PKV_OK;
}

PKV_API int pkv_block_free_count(const pkv_block_manager* mgr) {
    return mgr ? mgr->free_count : 0;
}

PKV_API int pkv_block_ref_count(const pkv_block_manager* mgr, int32_t block_id) {
    if (!mgr || block_id < 0 || block_id >= mgr->num_blocks) return -1;
    return mgr->ref[block_id];
}

PKV_API int pkv_block_free_ids(const pkv_block_manager* mgr, int32_t* out, int cap) {
    if (!mgr) return 0;
    int k = 0;
    for (int b = 0; b < mgr->num_blocks; ++b) {
        if (mgr->is_free(b)) {
            if (out && k < cap) out[k] = b;
            ++k;
        }
    }
    return k;
}

PKV_API pkv_status pkv_append_slots(pkv_block_manager* mgr, int32_t* block_tables,
                                    int max_blocks_per_seq, int32_t* context_lens, int num_seqs,
                                    int64_t* slot_mapping) {
    if (!mgr || num_seqs < 0 || max_blocks_per_seq < 0) return PKV_ERR_INVALID;
    if (num_seqs > 0 && (!block_tables || !context_lens || !slot_mapping)) return PKV_ERR_INVALID;
    const int B = mgr->block_size;
    pkv_status result = PKV_OK;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = context_lens[s];
        int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
        if (n < 0 || n / B > max_blocks_per_seq || (n % B != 0 && n / B >= max_blocks_per_seq)) {
            slot_mapping[s] = -1;
            result = PKV_ERR_NO_BLOCKS;
            continue;
        }
        const int j = n / B;
        if (n % B == 0) {
            // the last page is full (or there is none): open a new block
            if (j >= max_blocks_per_seq) {
                slot_mapping[s] = -1;
                result = PKV_ERR_NO_BLOCKS;
                continue;
            }
            int32_t b = -1;
            if (pkv_block_allocate(mgr, &b) != PKV_OK) {
                slot_mapping[s] = -1;
                result = PKV_ERR_NO_BLOCKS;
                continue;
            }
            row[j] = b;
        }
        slot_mapping[s] = (int64_t)row[j] * B + n % B;
        context_lens[s] = n + 1;
    }
    return result;
}

PKV_API pkv_status pkv_append_slots_cow(pkv_block_manager* mgr, int32_t* block_tables,
                                        int max_blocks_per_seq, int32_t* context_lens,
                                        int num_seqs, int64_t* slot_mapping,
                                        int64_t* copy_pairs, int* n_copy_pairs) {
    if (!mgr || num_seqs < 0 || max_blocks_per_seq < 0 || !n_copy_pairs) return PKV_ERR_INVALID;
    if (num_seqs > 0 && (!block_tables || !context_lens || !slot_mapping || !copy_pairs))
        return PKV_ERR_INVALID;
    const int B = mgr->block_size;
    pkv_status result = PKV_OK;
    int n_pairs = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = context_lens[s];
        int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
        const int j = n / B;
        if (n < 0 || j >= max_blocks_per_seq) {
            slot_mapping[s] = -1;
            result = PKV_ERR_NO_BLOCKS;
            continue;
        }
        if (n % B == 0) {
            // the last page is full (or there is none): open a new block
            int32_t b = -1;
            if (pkv_block_allocate(mgr, &b) != PKV_OK) {
                slot_mapping[s] = -1;
                result = PKV_ERR_NO_BLOCKS;
                continue;
            }
            row[j] = b;
        } else {
            const int32_t shared = row[j];
            if (shared < 0 || shared >= mgr->num_blocks) {
                slot_mapping[s] = -1;
                result = PKV_ERR_INVALID;
                continue;
            }
            if (mgr->ref[shared] > 1) {
                // the page is shared: write into a private copy instead
                int32_t b = -1;
                if (pkv_block_allocate(mgr, &b) != PKV_OK) {
                    slot_mapping[s] = -1;
                    result = PKV_ERR_NO_BLOCKS;
                    continue;
                }
                pkv_block_free(mgr, shared);
                row[j] = b;
                copy_pairs[2 * n_pairs] = shared;
                copy_pairs[2 * n_pairs + 1] = b;
                ++n_pairs;
            }
        }
        slot_mapping[s] = (int64_t)row[j] * B + n % B;
        context_lens[s] = n + 1;
    }
    *n_copy_pairs = n_pairs;
    return result;
}

PKV_API pkv_status pkv_defrag(pkv_block_manager* mgr, int32_t* block_tables,
                              int max_blocks_per_seq, int num_seqs, int64_t* pairs, int cap,
                              int* n_pairs) {
    if (!mgr || num_seqs < 0 || max_blocks_per_seq < 0 || cap < 0 || !n_pairs)
        return PKV_ERR_INVALID;
    if ((num_seqs > 0 && !block_tables) || (cap > 0 && !pairs)) return PKV_ERR_INVALID;
    const int nb = mgr->num_blocks;
    const int n_used = nb - mgr->free_count;
    // pair the used ids at or above n_used (increasing) with the free ids
    // below n_used (increasing)
    std::vector<int32_t> dst_of(nb, -1);
    int k = 0, hole = 0;
    for (int b = n_used; b < nb; ++b) {
        if (mgr->ref[b] == 0) continue;
        while (hole < n_used && mgr->ref[hole] != 0) ++hole;
        if (hole >= n_used) return PKV_ERR_INVALID;  // inconsistent counts
        if (k >= cap) {
            *n_pairs = k;
            return PKV_ERR_INVALID;                    // pairs buffer too small
        }
        pairs[2 * k] = b;
        pairs[2 * k + 1] = hole;
        dst_of[b] = hole;
        ++k;
        ++hole;
    }
    // move the counts and the free set, then repoint the tables
    for (int i = 0; i < k; ++i) {
        const int src = (int)pairs[2 * i], dst = (int)pairs[2 * i + 1];
        mgr->mark_held(dst);
        mgr->ref[dst] = mgr->ref[src];
        mgr->ref[src] = 0;
        mgr->mark_free(src);
    }
    for (int s = 0; s < num_seqs; ++s) {
        int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            if (row[j] >= 0 && row[j] < nb && dst_of[row[j]] >= 0) row[j] = dst_of[row[j]];
    }
    mgr->hint = 0;
    *n_pairs = k;
    return PKV_OK;
}

}  // extern "C"
