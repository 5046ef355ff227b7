"""Host-side block bookkeeping for the paged KV cache.

The device kernels never allocate blocks: the caller owns the pools and the
block tables, and this module is the caller-side free list. It follows
"Module 09: Efficient Attention", section "Paged Attention: The KV Cache as
Virtual Memory" (subsections "The Block Table" and "Code: A Paged KV Cache
from Scratch"): a free list hands out physical block ids, a sequence of n
tokens holds ceil(n / block_size) blocks and claims a new one whenever its
last block is full.
"""

import math

__all__ = [
    "blocks_needed",
    "paged_used_slots",
    "contiguous_reserved_slots",
    "BlockAllocator",
    "SequenceTables",
]


def blocks_needed(num_tokens, block_size):
    """ceil(num_tokens / block_size)."""
    return (num_tokens + block_size - 1) // block_size


def paged_used_slots(lengths, block_size):
    """Token slots held by paged sequences: whole blocks per sequence."""
    return sum(blocks_needed(n, block_size) * block_size for n in lengths)


def contiguous_reserved_slots(max_seq_len, num_sequences):
    """Token slots a contiguous scheme reserves up front."""
    return max_seq_len * num_sequences


class BlockAllocator:
    """Free list over ``num_blocks`` physical blocks, with reference counts.

    ``allocate()`` pops the most recently freed (or highest-numbered initial)
    block with one reference; ``share()`` adds a reference to an allocated
    block; ``free()`` drops one and returns the block to the free list when
    none is left. ``num_free + num_used`` never changes. An optional ``order``
    gives the initial free list (for example a shuffled permutation, so tables
    come out scattered).
    """

    def __init__(self, num_blocks, order=None):
        self.num_blocks = int(num_blocks)
        if order is None:
            self._free = list(range(self.num_blocks))
        else:
            self._free = [int(b) for b in order]
            if sorted(self._free) != list(range(self.num_blocks)):
                raise ValueError("order must be a permutation of range(num_blocks)")
        self._refs = {}

    @property
    def num_free(self):
        return len(self._free)

    @property
    def num_used(self):
        return len(self._refs)

    def refcount(self, blk):
        return self._refs.get(blk, 0)

    def allocate(self):
        if not self._free:
            raise MemoryError("no free KV blocks left")
        blk = self._free.pop()
        self._refs[blk] = 1
        return blk

    def share(self, blk):
        if blk not in self._refs:
            raise ValueError(f"block {blk} is not allocated")
        self._refs[blk] += 1
        return blk

    def free(self, blk):
        if blk not in self._refs:
            raise ValueError(f"block {blk} is not allocated")
        self._refs[blk] -= 1
        if self._refs[blk] == 0:
            del self._refs[blk]
            self._free.append(blk)


class SequenceTables:
    """Per-sequence block tables grown lazily through a :class:`BlockAllocator`.

    ``reserve(seq, new_len)`` claims blocks so that the sequence can hold
    ``new_len`` tokens (a new block exactly when the offset wraps to zero).
    ``release(seq)`` returns all of its blocks. ``as_rows(width)`` gives the
    rectangular int table the kernels read, padded with -1.
    """

    def __init__(self, allocator, block_size):
        self.allocator = allocator
        self.block_size = int(block_size)
        self.tables = {}
        self.lengths = {}

    def add_sequence(self):
        seq = len(self.tables)
        while seq in self.tables:
            seq += 1
        self.tables[seq] = []
        self.lengths[seq] = 0
        return seq

    def reserve(self, seq, new_len):
        need = blocks_needed(new_len, self.block_size)
        table = self.tables[seq]
        while len(table) < need:
            table.append(self.allocator.allocate())
        self.lengths[seq] = max(self.lengths[seq], new_len)
        return table

    def share_prefix(self, src, num_prefix_blocks):
        """A new sequence that points at the first ``num_prefix_blocks``
        blocks of ``src`` (no block is copied or allocated); it holds
        min(len(src), num_prefix_blocks * block_size) tokens."""
        blocks = self.tables[src][:num_prefix_blocks]
        if len(blocks) < num_prefix_blocks:
            raise ValueError("the source sequence has fewer blocks")
        seq = self.add_sequence()
        self.tables[seq] = [self.allocator.share(b) for b in blocks]
        self.lengths[seq] = min(self.lengths[src], num_prefix_blocks * self.block_size)
        return seq

    def prepare_write(self, seq, new_len):
        """Make positions [len(seq), new_len) writable: every block those
        positions fall in that another sequence still references is replaced
        by a private copy, then blocks are claimed up to ``new_len``. Returns
        the (source, destination) block pairs the device must copy first
        (``pa_copy_blocks``), in table order."""
        table = self.tables[seq]
        start = self.lengths[seq]
        copies = []
        if new_len > start:
            first = start // self.block_size
            last = min(blocks_needed(new_len, self.block_size), len(table))
            for i in range(first, last):
                old = table[i]
                if self.allocator.refcount(old) > 1:
                    new = self.allocator.allocate()
                    self.allocator.free(old)  # drops this sequence's reference
                    table[i] = new
                    copies.append((old, new))
        self.reserve(seq, new_len)
        return copies

    def release(self, seq):
        for blk in self.tables.pop(seq):
            self.allocator.free(blk)
        self.lengths.pop(seq)

    def as_rows(self, seqs, width=None):
        rows = [list(self.tables[s]) for s in seqs]
        if width is None:
            width = max((len(r) for r in rows), default=0)
        width = max(width, 1)
        out = []
        for r in rows:
            if len(r) > width:
                raise ValueError("block table wider than the requested width")
            out.append(r + [-1] * (width - len(r)))
        return out

    @staticmethod
    def waste(lengths, block_size):
        """Unused slots in the last, partially filled block of each sequence."""
        return sum(blocks_needed(n, block_size) * block_size - n for n in lengths)

    @staticmethod
    def max_context(free_bytes, bytes_per_token):
        """Tokens that fit in ``free_bytes`` of cache memory."""
        return math.floor(free_bytes / bytes_per_token)
