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

Prefix caching ("PagedAttention por dentro", section "Prefix caching
cross-session"; "Cómo funciona realmente vLLM", section "Automatic Prefix
Caching": finished requests' blocks are indexed by a hash of their content and
reused by a new request that begins the same way).  Reading: a full block's
K/V depend on every token up to it, so its key chains over the whole prefix:
    key_j = FNV1a64(le64(key_{j-1}) || le32(tokens[16j .. 16j+15])), key_{-1} = 0
(FNV-1a, 64 bits: offset basis 0xcbf29ce484222325, prime 0x100000001b3).
A lookup matches a cached block only if its key and its own 16 tokens agree.
Released blocks that carry a key wait in an evictable list (least recently
released first) and are reused only when the free list is empty; taking one
drops its key.
"""
from __future__ import annotations

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a of a byte string."""
    h = FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_key(parent_key: int, tokens) -> int:
    """Key of a full block given its parent's key (0 for the first block)."""
    data = int(parent_key & MASK64).to_bytes(8, "little")
    for t in tokens:
        data += int(t & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


def block_keys(tokens, block_size: int = 16):
    """Keys of the full blocks of a token sequence."""
    keys, parent = [], 0
    for j in range(len(tokens) // block_size):
        parent = block_key(parent, tokens[j * block_size:(j + 1) * block_size])
        keys.append(parent)
    return keys


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
        # prefix cache
        self.cached: dict[int, int] = {}          # key -> block
        self.block_key: dict[int, int] = {}       # block -> key
        self.block_tokens: dict[int, tuple] = {}  # block -> its 16 tokens
        self.evictable: list[int] = []            # released keyed blocks, oldest first
        self.swapped: set[int] = set()            # sequences whose blocks are swapped out

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
    def num_evictable(self) -> int:
        return len(self.evictable)

    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.evictable:
            b = self.evictable.pop(0)
            key = self.block_key.pop(b)
            del self.cached[key]
            del self.block_tokens[b]
        else:
            raise NoBlocks()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            if b in self.block_key:
                self.evictable.append(b)
            else:
                self.free.append(b)

    def _live(self, seq: int) -> None:
        if seq in self.swapped:
            raise ValueError("sequence is swapped out")

    def alloc_seq_cached(self, seq: int, tokens) -> int:
        """New sequence holding ``tokens``: its leading full blocks are taken from the
        prefix cache where they match; returns how many tokens were found cached."""
        if seq in self.tables:
            raise ValueError("sequence exists")
        n = len(tokens)
        hits = []
        parent = 0
        for j in range(n // self.block_size):
            own = tuple(int(t) for t in tokens[j * self.block_size:(j + 1) * self.block_size])
            parent = block_key(parent, own)
            b = self.cached.get(parent)
            if b is None or self.block_tokens[b] != own:
                break
            hits.append(b)
        need = self.blocks_needed(n) - len(hits)
        reusable = sum(1 for b in hits if self.ref[b] == 0)
        if need > len(self.free) + len(self.evictable) - reusable:
            raise NoBlocks()
        for b in hits:
            if self.ref[b] == 0:
                self.evictable.remove(b)
            self.ref[b] += 1
        table = list(hits) + [self._take() for _ in range(need)]
        self.tables[seq] = table
        self.tokens[seq] = n
        return len(hits) * self.block_size

    def register_prefix(self, seq: int, tokens) -> int:
        """Index the sequence's full blocks by key (their K/V are now written);
        returns how many blocks were newly indexed."""
        table = self.tables[seq]
        self._live(seq)
        n = min(len(tokens), self.tokens[seq])
        added, parent = 0, 0
        for j in range(n // self.block_size):
            own = tuple(int(t) for t in tokens[j * self.block_size:(j + 1) * self.block_size])
            parent = block_key(parent, own)
            b = table[j]
            if b < 0 or parent in self.cached or b in self.block_key:
                continue
            self.cached[parent] = b
            self.block_key[b] = parent
            self.block_tokens[b] = own
            added += 1
        return added

    def alloc_seq(self, seq: int, num_tokens: int) -> list[int]:
        """Give a new sequence room for ``num_tokens`` tokens (all or nothing)."""
        if seq in self.tables or num_tokens < 0:
            raise ValueError("sequence exists or bad length")
        need = self.blocks_needed(num_tokens)
        if need > len(self.free) + len(self.evictable):
            raise NoBlocks()
        self.tables[seq] = [self._take() for _ in range(need)]
        self.tokens[seq] = num_tokens
        return self.table(seq)

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (reference counts + 1)."""
        if parent not in self.tables or child in self.tables:
            raise ValueError("bad fork")
        self._live(parent)
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = self.tokens[parent]
        for b in self.tables[child]:
            if b >= 0:
                self.ref[b] += 1

    def make_private(self, seq: int, logical_block: int):
        """Copy-on-write of one logical block; returns (src, dst) or None if private."""
        table = self.tables[seq]
        self._live(seq)
        old = table[logical_block]
        if old < 0:
            raise ValueError("block released by trim_window")
        if self.ref[old] <= 1:
            # private already; a block the prefix cache indexes is about to be
            # written in place, so its content stops matching its key: drop it
            if old in self.block_key:
                del self.cached[self.block_key.pop(old)]
                del self.block_tokens[old]
            return None
        new = self._take()
        self.ref[old] -= 1        # still held by another sequence: stays > 0
        table[logical_block] = new
        return (old, new)

    def append_slot(self, seq: int):
        """Room for one more token.  Returns (slot, cow) where cow is (src, dst) or None."""
        table = self.tables[seq]
        self._live(seq)
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
        self.swapped.discard(seq)
        for b in reversed(table):
            if b >= 0:
                self._release(b)

    def trim_window(self, seq: int, window: int) -> int:
        """Sliding window ("PagedAttention por dentro", section "Sliding window
        attention": only the active window's blocks are kept).  Blocks whose
        positions all precede N - window are released, last first, and their
        entries become -1; returns how many were released."""
        if window <= 0 or seq not in self.tables:
            raise ValueError("bad trim")
        table = self.tables[seq]
        self._live(seq)
        n = self.tokens[seq]
        dead = (n - window) // self.block_size if n > window else 0
        released = 0
        for j in range(dead - 1, -1, -1):
            if table[j] >= 0:
                self._release(table[j])
                table[j] = -1
                released += 1
        return released

    def swap_out(self, seq: int) -> list[int]:
        """Preemption by swap ("PagedAttention por dentro", section "Evicción y
        preemption"): returns the sequence's blocks in table order, releases them
        (last entry first) and marks their entries -2."""
        table = self.tables[seq]
        self._live(seq)
        ids = [b for b in table if b >= 0]
        for j in range(len(table) - 1, -1, -1):
            if table[j] >= 0:
                self._release(table[j])
                table[j] = -2
        self.swapped.add(seq)
        return ids

    def swap_in(self, seq: int) -> list[int]:
        """Fresh private blocks for the -2 entries, in table order (all or nothing)."""
        if seq not in self.swapped:
            raise ValueError("sequence is not swapped out")
        table = self.tables[seq]
        need = sum(1 for b in table if b == -2)
        if need > len(self.free) + len(self.evictable):
            raise NoBlocks()
        ids = []
        for j, b in enumerate(table):
            if b == -2:
                table[j] = self._take()
                ids.append(table[j])
        self.swapped.discard(seq)
        return ids

    # -- occupancy -------------------------------------------------------
    def stats(self) -> dict:
        """Pool occupancy and internal fragmentation ("Cómo funciona realmente
        vLLM", section "La sobre-reserva estática y los tres tipos de
        desperdicio": slots reserved for a sequence that never get a token).
        Sequence s with N tokens holds min(16, N - 16 j) tokens in the block of
        its table entry j; a block shared by several entries holds the most of
        them (each fills it from offset 0)."""
        bs = self.block_size
        held = {}
        logical = 0
        for seq, table in self.tables.items():
            n = self.tokens[seq]
            for j, b in enumerate(table):
                if b < 0:
                    continue
                k = min(bs, n - j * bs)
                logical += k
                held[b] = max(held.get(b, 0), k)
        used = sum(1 for r in self.ref if r >= 1)
        reserved = used * bs
        filled = sum(held.values())
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": len(self.free),
            "evictable_blocks": len(self.evictable),
            "used_blocks": used,
            "shared_blocks": sum(1 for r in self.ref if r >= 2),
            "reserved_slots": reserved,
            "filled_slots": filled,
            "logical_tokens": logical,
            "internal_fragmentation": (reserved - filled) / reserved if reserved else 0.0,
        }

    # -- invariants ------------------------------------------------------
    def check(self) -> None:
        counted = [0] * self.num_blocks
        for seq, table in self.tables.items():
            assert len(table) == self.blocks_needed(self.tokens[seq])
            for b in table:
                if b >= 0:
                    counted[b] += 1
        assert counted == self.ref
        free = set(self.free)
        ev = set(self.evictable)
        assert len(free) == len(self.free) and len(ev) == len(self.evictable)
        assert not (free & ev)
        for b in range(self.num_blocks):
            assert (b in free or b in ev) == (self.ref[b] == 0)
            assert (b in ev) <= (b in self.block_key)
        for key, b in self.cached.items():
            assert self.block_key[b] == key
