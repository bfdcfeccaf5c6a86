"""Plain-Python restatement of the block allocator and scheduler that the page
"大模型长文本推理基座从 FlashAttention 硬件加速机制到 vLLM 核心 PagedAttention
显存物理布局深度剖析" gives in its section 三 (PhysicalBlock, KVBlockManager,
BlockTable, PagedAttentionScheduler), used as the oracle for the library's
native block manager.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.

The page's text lost several operators in extraction.  Readings taken (the
only ones the surrounding code and its comments support):
  * ``is_free``: ``ref_count == 0``;
  * ``allocate``: ``free_blocks.pop(0)`` then ``ref_count = 1``;
  * ``free``: ``if ref_count > 0: ref_count -= 1``; when it reaches 0 the id
    goes back to the free list, which is kept sorted so that the lowest id
    is handed out first;
  * ``add_reference``: ``ref_count += 1``;
  * ``register_request``: ``ceil(prompt_len / block_size)`` blocks;
  * ``append_token``: a new block when ``num_allocated_tokens % block_size ==
    0``, then ``num_allocated_tokens += 1``; an empty pool makes the append
    fail (return False) without changing the table.

Parity: pinned by the page's own walkthrough (tests/golden/allocator_walkthrough.json).
"""
from __future__ import annotations


class OutOfBlocks(MemoryError):
    """Raised by ``allocate`` when no physical block is free (the page raises
    MemoryError with a "CUDA Out of Memory" message)."""


class PhysicalBlock:
    def __init__(self, block_id: int, block_size: int = 16):
        self.block_id = block_id
        self.block_size = block_size
        self.ref_count = 0

    def is_free(self) -> bool:
        return self.ref_count == 0


class KVBlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, free_ids=None):
        self.block_size = block_size
        self.gpu_blocks = [PhysicalBlock(i, block_size) for i in range(num_blocks)]
        if free_ids is None:
            self.free_blocks = list(range(num_blocks))
        else:
            # A pool that starts part-used: ids not listed are held once.
            self.free_blocks = sorted(int(i) for i in free_ids)
            held = set(range(num_blocks)) - set(self.free_blocks)
            for i in held:
                self.gpu_blocks[i].ref_count = 1

    def allocate(self) -> int:
        if not self.free_blocks:
            raise OutOfBlocks("CUDA Out of Memory: No free physical blocks available in pool!")
        block_id = self.free_blocks.pop(0)
        self.gpu_blocks[block_id].ref_count = 1
        return block_id

    def free(self, block_id: int) -> None:
        block = self.gpu_blocks[block_id]
        if block.ref_count > 0:
            block.ref_count -= 1
            if block.ref_count == 0:
                self.free_blocks.append(block_id)
                self.free_blocks.sort()

    def add_reference(self, block_id: int) -> None:
        self.gpu_blocks[block_id].ref_count += 1

    def get_free_blocks_count(self) -> int:
        return len(self.free_blocks)


class BlockTable:
    def __init__(self, request_id):
        self.request_id = request_id
        self.physical_block_ids: list[int] = []
        self.num_allocated_tokens = 0


class PagedAttentionScheduler:
    def __init__(self, num_blocks: int = 10, block_size: int = 16, free_ids=None):
        self.manager = KVBlockManager(num_blocks, block_size, free_ids)
        self.block_size = block_size
        self.active_requests: dict = {}

    def register_request(self, request_id, prompt_len: int) -> BlockTable:
        table = BlockTable(request_id)
        required_blocks = (prompt_len + self.block_size - 1) // self.block_size
        for _ in range(required_blocks):
            table.physical_block_ids.append(self.manager.allocate())
        table.num_allocated_tokens = prompt_len
        self.active_requests[request_id] = table
        return table

    def adopt(self, request_id, block_ids, num_tokens: int) -> BlockTable:
        """Install an existing table (blocks already held) without allocating;
        used to start from a generated cache state."""
        table = BlockTable(request_id)
        table.physical_block_ids = [int(b) for b in block_ids]
        table.num_allocated_tokens = int(num_tokens)
        self.active_requests[request_id] = table
        return table

    def append_token(self, request_id) -> bool:
        table = self.active_requests.get(request_id)
        if not table:
            return False
        current_tokens = table.num_allocated_tokens
        if current_tokens % self.block_size == 0:
            try:
                new_block_id = self.manager.allocate()
            except OutOfBlocks:
                return False
            table.physical_block_ids.append(new_block_id)
        table.num_allocated_tokens += 1
        return True

    def finish_request(self, request_id) -> None:
        table = self.active_requests.pop(request_id, None)
        if table:
            for block_id in table.physical_block_ids:
                self.manager.free(block_id)


def append_slots_cow(tables, context_lens, block_size: int, free_ids, num_blocks: int,
                     ref_counts):
    """append_slots with copy-on-write ([LAYOUT] section 四.2): several
    requests may point at one physical block (ref_count > 1).  The page
    says only a request that writes its own next token into such a block
    triggers the copy: it gets a freshly allocated private block holding a
    copy of the shared one, and drops its reference to the shared block.

    Readings: the copy happens when the token's page is an existing shared
    block (a partly filled last page; a full page opens a new block as in
    append_token).  ref_counts gives the starting count of every block
    (free ids have 0).  Returns (new_tables, new_lens, slots, copy_pairs,
    free_after, ref_after); copy_pairs lists (shared block, private block)
    in sequence order, for the caller to copy before writing.
    """
    mgr = KVBlockManager(num_blocks, block_size, free_ids)
    for b in range(num_blocks):
        mgr.gpu_blocks[b].ref_count = int(ref_counts[b])
    tables = [list(map(int, t)) for t in tables]
    lens = [int(n) for n in context_lens]
    slots, pairs = [], []
    for s in range(len(tables)):
        n = lens[s]
        j = n // block_size
        if n % block_size == 0:
            try:
                tables[s].append(mgr.allocate())
            except OutOfBlocks:
                slots.append(-1)
                continue
        else:
            b = tables[s][j]
            if mgr.gpu_blocks[b].ref_count > 1:
                try:
                    nb = mgr.allocate()
                except OutOfBlocks:
                    slots.append(-1)
                    continue
                mgr.free(b)
                tables[s][j] = nb
                pairs.append((b, nb))
        slots.append(tables[s][j] * block_size + n % block_size)
        lens[s] = n + 1
    refs = [blk.ref_count for blk in mgr.gpu_blocks]
    return tables, lens, slots, pairs, list(mgr.free_blocks), refs


def append_slots(tables, context_lens, block_size: int, free_ids, num_blocks: int):
    """One decode step's append for every sequence, in sequence order: each
    sequence gets one new token through ``append_token`` (a new block from the
    free list when its last page is full) and the flat slot that token is
    written to, ``table[n // B] * B + n % B`` for its old length n.  A
    sequence whose append fails gets slot -1.

    Returns (new_tables (list of lists), new_lens, slots, free_ids_after).
    """
    sch = PagedAttentionScheduler(num_blocks, block_size, free_ids)
    for s, (ids, n) in enumerate(zip(tables, context_lens)):
        sch.adopt(s, ids, n)
    slots = []
    for s in range(len(tables)):
        n = sch.active_requests[s].num_allocated_tokens
        ok = sch.append_token(s)
        if not ok:
            slots.append(-1)
            continue
        ids = sch.active_requests[s].physical_block_ids
        slots.append(ids[n // block_size] * block_size + n % block_size)
    new_tables = [list(sch.active_requests[s].physical_block_ids) for s in range(len(tables))]
    new_lens = [sch.active_requests[s].num_allocated_tokens for s in range(len(tables))]
    return new_tables, new_lens, slots, list(sch.manager.free_blocks)


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
