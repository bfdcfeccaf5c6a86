"""Block allocator rules of paged KV caching, restated as plain functions over
a reference-count list; the oracle for the library's native block manager
(host and device).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.

The rules, as the page "大模型长文本推理基座从 FlashAttention 硬件加速机制到
vLLM 核心 PagedAttention 显存物理布局深度剖析" states them in its section 二.2
(logical blocks of 16 tokens mapped to physical blocks by a block table)
and section 三 (a pool of physical blocks with reference counts; a request
gets blocks for its prompt, one more each time its last block is full, and
gives them back when it finishes):

  R1  The pool holds ids 0 .. N-1.  Each id carries a reference count; an id
      whose count is 0 is free.
  R2  Taking a block hands out the lowest free id and sets its count to 1
      (the page keeps its free list sorted and takes the first entry).  With
      no free id the take fails.
  R3  Dropping a reference lowers a held id's count by one; at 0 the id is
      free again (a free id stays free).
  R4  Sharing a held block (a common prompt prefix, a forked request) adds a
      reference.  Sharing a free id is refused (the page's code would allow
      it while leaving the id in its free list; that state is never valid).
  R5  A request of n tokens holds ceil(n / B) blocks.  Its token number n
      (0-based) needs a new block exactly when n mod B == 0; if the take
      fails the token is not added and the request is unchanged.
  R6  Token n of a request lives at row n mod B of its logical block n div B,
      i.e. at flat slot table[n div B] * B + n mod B of the pool.

Here a pool is a list of reference counts; a request is its table (list of
physical ids) and its token count.  Readings where the extracted page text
is garbled (lost comparison and update operators) are listed in the repo's
design notes; the two-request walkthrough of section 三 pins the result
(tests/golden/allocator_walkthrough.json).
"""
from __future__ import annotations


# ------------------------------------------------------------------ pool

def make_pool(num_blocks: int, free_ids=None) -> list[int]:
    """R1: reference counts of a pool of num_blocks ids.  With free_ids
    given, the ids not listed start held once (a pool already in use)."""
    if free_ids is None:
        return [0] * num_blocks
    refs = [1] * num_blocks
    for b in free_ids:
        refs[int(b)] = 0
    return refs


def free_list(refs) -> list[int]:
    """The free ids in increasing order (the order R2 hands them out)."""
    return [b for b, r in enumerate(refs) if r == 0]


def take_block(refs):
    """R2: the lowest free id, now held once; None if every id is held."""
    for b, r in enumerate(refs):
        if r == 0:
            refs[b] = 1
            return b
    return None


def drop_reference(refs, b: int) -> None:
    """R3: one reference fewer on block b (nothing happens to a free id)."""
    if refs[b] > 0:
        refs[b] -= 1


def share_block(refs, b: int) -> None:
    """R4: one reference more on the held block b."""
    if refs[b] <= 0:
        raise ValueError(f"block {b} is free and cannot be shared")
    refs[b] += 1


# -------------------------------------------------------------- requests

def blocks_needed(num_tokens: int, block_size: int) -> int:
    """R5: blocks a request of num_tokens tokens holds."""
    return -(-num_tokens // block_size)


def admit(refs, num_tokens: int, block_size: int):
    """A new request with a prompt of num_tokens tokens: its table of
    blocks_needed blocks taken one after another (R2), or None when the
    pool runs out (the blocks taken so far are given back)."""
    table = []
    for _ in range(blocks_needed(num_tokens, block_size)):
        b = take_block(refs)
        if b is None:
            for t in table:
                drop_reference(refs, t)
            return None
        table.append(b)
    return table


def slot_of(table, n: int, block_size: int) -> int:
    """R6: flat pool slot of token n."""
    return table[n // block_size] * block_size + n % block_size


def add_token(refs, table, num_tokens: int, block_size: int):
    """R5 for one request: returns (slot of the new token, new token count),
    or (-1, num_tokens) when a new block was needed and none was free.
    `table` grows in place when a block is opened."""
    if num_tokens % block_size == 0:
        b = take_block(refs)
        if b is None:
            return -1, num_tokens
        table.append(b)
    return slot_of(table, num_tokens, block_size), num_tokens + 1


def release(refs, table) -> None:
    """A finished request gives back one reference on each of its blocks."""
    for b in table:
        drop_reference(refs, b)


# ------------------------------------------------------- one decode step

def append_slots(tables, context_lens, block_size: int, free_ids, num_blocks: int):
    """One decode step's append for every sequence, in sequence order: each
    sequence gets one new token (add_token), starting from a pool whose free
    ids are `free_ids` and whose other ids are held once.

    Returns (new_tables, new_lens, slots, free_ids_after); a sequence whose
    append failed has slot -1 and keeps its table and length."""
    refs = make_pool(num_blocks, free_ids)
    new_tables = [[int(b) for b in t] for t in tables]
    new_lens, slots = [], []
    for table, n in zip(new_tables, context_lens):
        slot, n_after = add_token(refs, table, int(n), block_size)
        slots.append(slot)
        new_lens.append(n_after)
    return new_tables, new_lens, slots, free_list(refs)


def append_slots_cow(tables, context_lens, block_size: int, free_ids, num_blocks: int,
                     ref_counts):
    """append_slots with copy-on-write ([LAYOUT] section 四.2): several
    requests may point at one physical block (count > 1), and a request
    that writes its next token into such a shared block first gets a
    private copy: a newly taken block that replaces the shared one in its
    table, the shared block losing that reference.

    Readings: the copy happens only when the token's page is an existing
    block held more than once (a partly filled last page); a token that
    starts a page opens a new block as in add_token.  ref_counts gives every
    block's starting count (free ids 0; free_ids must list exactly those).
    Returns (new_tables, new_lens, slots, copy_pairs, free_after, ref_after);
    copy_pairs lists (shared block, private block) in sequence order, for
    the caller to copy before the tokens are written."""
    refs = [int(r) for r in ref_counts]
    assert free_list(refs) == sorted(int(b) for b in free_ids)
    assert len(refs) == num_blocks
    new_tables = [[int(b) for b in t] for t in tables]
    new_lens, slots, pairs = [], [], []
    for table, n in zip(new_tables, context_lens):
        n = int(n)
        j = n // block_size
        if n % block_size != 0 and refs[table[j]] > 1:
            private = take_block(refs)
            if private is None:
                slots.append(-1)
                new_lens.append(n)
                continue
            pairs.append((table[j], private))
            drop_reference(refs, table[j])
            table[j] = private
        slot, n_after = add_token(refs, table, n, block_size)
        slots.append(slot)
        new_lens.append(n_after)
    return new_tables, new_lens, slots, pairs, free_list(refs), refs


# ----------------------------------------------------- defragmentation

def defrag_plan(ref_counts):
    """Defragmentation by block copies ("vLLM 中 FlashAttention 与 KVCache 交换
    机制深度解析": swap_blocks also serves to rearrange scattered pages into a
    more compact layout).  Reading: with n blocks in use, every used block
    whose id is >= n moves to a free id < n, the lowest used ids outside
    going to the lowest free ids inside, so that afterwards the used blocks
    are exactly [0, n).  Returns the (source, destination) pairs."""
    nb = len(ref_counts)
    used = [b for b in range(nb) if ref_counts[b] > 0]
    n = len(used)
    holes = [b for b in range(n) if ref_counts[b] == 0]
    movers = [b for b in used if b >= n]
    assert len(holes) == len(movers)
    return list(zip(movers, holes))


def apply_defrag(tables, ref_counts, pairs):
    """Tables and reference counts after the pairs' blocks moved."""
    where = dict(pairs)
    new_tables = [[where.get(b, b) for b in t] for t in tables]
    refs = list(ref_counts)
    for src, dst in pairs:
        refs[dst], refs[src] = refs[src], 0
    return new_tables, refs
