"""Plain-Python model of the paged KV block manager.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It restates the block
bookkeeping of "PagedAttention por dentro: bloques, tabla de páginas, evicción
y el estado del arte del KV cache en 2026":

* "La tabla de páginas (block table)": every sequence owns an ordered list of
  physical block ids; when the sequence already holds N tokens, its next token
  goes into the last block if N mod 16 != 0, otherwise a new block is taken
  from the global pool and appended.  Freeing a sequence returns its blocks.
* "El pool de bloques": one global pool of fixed-size blocks shared by all
  sequences.
* "Copy-on-write para sampling paralelo": forked sequences share their blocks
  (reference counts); a sequence about to modify a shared block first gets a
  private copy of that one block.

Deterministic allocation policy (a contract the native block manager follows
as well): the free list is a stack that initially pops 0, 1, 2, ...; a freed
block is pushed back and is the next one handed out.  ``free_seq`` releases a
table from its last entry to its first, so the first block of the freed table
is reused first.
"""
from __future__ import annotations


class NoBlocks(Exception):
    """The pool has no free block for the request (nothing was changed)."""


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int = 16):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool geometry")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks - 1, -1, -1))  # pop() yields 0, 1, 2, ...
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.tokens: dict[int, int] = {}

    # -- queries ---------------------------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def num_tokens(self, seq: int) -> int:
        return self.tokens[seq]

    def ref_count(self, block: int) -> int:
        return self.ref[block]

    def blocks_needed(self, num_tokens: int) -> int:
        return -(-num_tokens // self.block_size)

    # -- mutations -------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise NoBlocks()
        b = self.free.pop()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def alloc_seq(self, seq: int, num_tokens: int) -> list[int]:
        """Give a new sequence room for ``num_tokens`` tokens (all or nothing)."""
        if seq in self.tables or num_tokens < 0:
            raise ValueError("sequence exists or bad length")
        need = self.blocks_needed(num_tokens)
        if need > len(self.free):
            raise NoBlocks()
        self.tables[seq] = [self._take() for _ in range(need)]
        self.tokens[seq] = num_tokens
        return self.table(seq)

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (reference counts + 1)."""
        if parent not in self.tables or child in self.tables:
            raise ValueError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def make_private(self, seq: int, logical_block: int):
        """Copy-on-write of one logical block; returns (src, dst) or None if private."""
        table = self.tables[seq]
        old = table[logical_block]
        if self.ref[old] <= 1:
            return None
        new = self._take()
        self.ref[old] -= 1
        table[logical_block] = new
        return (old, new)

    def append_slot(self, seq: int):
        """Room for one more token.  Returns (slot, cow) where cow is (src, dst) or None."""
        table = self.tables[seq]
        n = self.tokens[seq]
        cow = None
        if n % self.block_size == 0:
            table.append(self._take())
        else:
            cow = self.make_private(seq, len(table) - 1)
        slot = table[n // self.block_size] * self.block_size + n % self.block_size
        self.tokens[seq] = n + 1
        return slot, cow

    def free_seq(self, seq: int) -> None:
        table = self.tables.pop(seq)
        del self.tokens[seq]
        for b in reversed(table):
            self.ref[b] -= 1
            assert self.ref[b] >= 0
            if self.ref[b] == 0:
                self.free.append(b)

    # -- invariants ------------------------------------------------------
    def check(self) -> None:
        counted = [0] * self.num_blocks
        for seq, table in self.tables.items():
            assert len(table) == self.blocks_needed(self.tokens[seq])
            for b in table:
                counted[b] += 1
        assert counted == self.ref
        free = set(self.free)
        assert len(free) == len(self.free)
        for b in range(self.num_blocks):
            assert (b in free) == (self.ref[b] == 0)
