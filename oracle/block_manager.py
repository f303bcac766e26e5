"""Reference model of the paged-KV block manager.

TEST INFRASTRUCTURE ONLY (see the package docstring): the native block
manager of the library is checked against this model operation by operation.

What it models ("paged-attention-runtime" summary, CORE CAPABILITIES 1:
fixed 16-token blocks, free-list allocator, reference counting, prefix
sharing, copy-on-write, fragmentation metrics; "PagedAttention & KV-Cache
Memory Management": the logical-to-physical allocator with a prefix cache
keyed by content hash, and section 4.1.1, page-level reference counts with a
fresh page and a copy when a shared page diverges):

* physical blocks 0 .. n-1, each with a reference count, the number of
  tokens it holds (its fill) and the prefix hash it is registered under;
* a free list used as a stack: initially it hands out 0, 1, 2, ...; a freed
  block goes on top and is handed out next;
* ``allocate(hashes)``: one block per entry.  An entry with a hash already in
  the prefix cache shares that block (its count goes up by one); any other
  entry takes a free block (count 1) and, if it has a hash, registers it.
  All-or-nothing: if the free list cannot serve every entry that needs a
  fresh block, nothing changes and ``None`` is returned;
* ``free(ids)``: one reference dropped per id; a block whose count reaches 0
  loses its hash registration and its fill and goes back on the free list;
* ``fork(ids)``: one reference added per id (a second sequence or beam now
  points at the block);
* ``cow(id)``: called before writing into a block.  If others share it
  (count > 1) a fresh block is taken, the old block loses one reference, the
  new one gets count 1 and the old block's fill, and the caller copies the
  contents (the returned flag).  An unshared block is returned as it is.  The
  block that will be written is not (or no longer) registered under a prefix
  hash, since its contents are about to change;
* ``set_fill(ids, tokens)``: the number of valid tokens in each block;
* ``stats()``: free, used (count > 0), shared (count > 1) and logical
  (sum of counts) blocks, stored tokens, internal fragmentation
  1 - tokens / (used * block_size) and sharing saving 1 - used / logical.
"""
from __future__ import annotations

NO_HASH = 0  # hash value meaning "no prefix hash" (hashes are uint64)


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int = 16):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad sizes")
        self.block_size = block_size
        self.refcnt = [0] * num_blocks
        self.fill = [0] * num_blocks
        self.hash_of = [NO_HASH] * num_blocks
        self.free_list = list(range(num_blocks - 1, -1, -1))  # top = end
        self.cache: dict[int, int] = {}

    # ------------------------------------------------------------ queries
    @property
    def num_blocks(self) -> int:
        return len(self.refcnt)

    def num_free(self) -> int:
        return len(self.free_list)

    # ---------------------------------------------------------- operations
    def allocate(self, hashes):
        """Returns the list of block ids, or None (nothing changed)."""
        hashes = [int(h) for h in hashes]
        # entries that need a fresh block: no hash, or a hash neither cached
        # nor introduced by an earlier entry of this call
        seen = set()
        fresh = 0
        for h in hashes:
            if h != NO_HASH and (h in self.cache or h in seen):
                continue
            fresh += 1
            if h != NO_HASH:
                seen.add(h)
        if fresh > len(self.free_list):
            return None
        ids = []
        for h in hashes:
            if h != NO_HASH and h in self.cache:
                b = self.cache[h]
                self.refcnt[b] += 1
            else:
                b = self.free_list.pop()
                self.refcnt[b] = 1
                self.fill[b] = 0
                self.hash_of[b] = h
                if h != NO_HASH:
                    self.cache[h] = b
            ids.append(b)
        return ids

    def _check_ids(self, ids):
        for b in ids:
            if not 0 <= b < self.num_blocks or self.refcnt[b] <= 0:
                return False
        return True

    def free(self, ids) -> bool:
        """Drop one reference per id; False (nothing changed) if an id is not
        a block in use or is listed more times than it has references."""
        ids = [int(b) for b in ids]
        if not self._check_ids(ids):
            return False
        need = {}
        for b in ids:
            need[b] = need.get(b, 0) + 1
        if any(need[b] > self.refcnt[b] for b in need):
            return False
        for b in ids:
            self.refcnt[b] -= 1
            if self.refcnt[b] == 0:
                h = self.hash_of[b]
                if h != NO_HASH and self.cache.get(h) == b:
                    del self.cache[h]
                self.hash_of[b] = NO_HASH
                self.fill[b] = 0
                self.free_list.append(b)
        return True

    def fork(self, ids) -> bool:
        ids = [int(b) for b in ids]
        if not self._check_ids(ids):
            return False
        for b in ids:
            self.refcnt[b] += 1
        return True

    def cow(self, b: int):
        """Returns (block to write, copy needed) or None if b is not in use
        or no free block is left for the copy (nothing changed)."""
        b = int(b)
        if not self._check_ids([b]):
            return None
        if self.refcnt[b] == 1:
            h = self.hash_of[b]
            if h != NO_HASH and self.cache.get(h) == b:
                del self.cache[h]
            self.hash_of[b] = NO_HASH
            return b, False
        if not self.free_list:
            return None
        n = self.free_list.pop()
        self.refcnt[b] -= 1
        self.refcnt[n] = 1
        self.fill[n] = self.fill[b]
        self.hash_of[n] = NO_HASH
        return n, True

    def cow_batch(self, ids):
        """``cow`` of each id in order, all-or-nothing: returns (blocks to
        write, [(source, copy)] pairs) or None (nothing changed)."""
        ids = [int(b) for b in ids]
        if not self._check_ids(ids):
            return None
        left, copies = {}, 0
        for b in ids:
            c = left.setdefault(b, self.refcnt[b])
            if c > 1:
                left[b] = c - 1
                copies += 1
        if copies > len(self.free_list):
            return None
        out, pairs = [], []
        for b in ids:
            nb, copied = self.cow(b)
            out.append(nb)
            if copied:
                pairs.append((b, nb))
        return out, pairs

    def set_fill(self, ids, tokens) -> bool:
        ids = [int(b) for b in ids]
        tokens = [int(t) for t in tokens]
        if not self._check_ids(ids) or any(not 0 <= t <= self.block_size for t in tokens):
            return False
        for b, t in zip(ids, tokens):
            self.fill[b] = t
        return True

    def stats(self):
        used = sum(1 for r in self.refcnt if r > 0)
        shared = sum(1 for r in self.refcnt if r > 1)
        logical = sum(self.refcnt)
        tokens = sum(f for f, r in zip(self.fill, self.refcnt) if r > 0)
        frag = 1.0 - tokens / (used * self.block_size) if used else 0.0
        saving = 1.0 - used / logical if logical else 0.0
        return {"free": len(self.free_list), "used": used, "shared": shared,
                "logical": logical, "tokens": tokens, "internal_fragmentation": frag,
                "sharing_saving": saving}


def blocks_for_tokens(tokens: int, block_size: int = 16) -> int:
    """Blocks a sequence of `tokens` tokens occupies (whole blocks)."""
    return (int(tokens) + block_size - 1) // block_size
