"""Model of the pages' host block manager, used to check the product's manager.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it follows, by page title and section:
  [PidokuInfra 10]  "10 PagedAttention", section 4 "Tiny example": a stack of
                    free block ids; Allocate(n) takes the top n entries in
                    slice order and sets their refcount to 1, or fails with no
                    state change when fewer than n are free; Free decrements
                    each refcount and pushes a block back only when it reaches
                    0; Fork increments every refcount and copies the table;
                    BlocksNeeded = ceil(tokens / B); a sequence grows by one
                    block when a token crosses a block boundary;
                    PhysicalIndex = table[pos / B] * B + pos % B.
  [nano-vLLM ch.04] "04 · PagedAttention", section 6 "Copy-on-write block
                    sharing" and section 7 "The BlockManager in code": before a
                    write into a block whose refcount is above 1, copy it,
                    decrement the old block's refcount and give the copy to
                    the writer; with refcount 1, write in place.
  [tokentrails]     "PagedAttention", step 4: only a partly filled shared block
                    is ever written, so only such a block is copied.

Prefix caching ([PidokuInfra 10] section 5 "The relationship to prefix
caching"; [nano-vLLM ch.04] section 7, hash_to_block): the token ids of each
full block are hashed and kept in a hash -> block map; a new sequence whose
first blocks hash to existing blocks points at them (refcount + 1) instead of
computing them.

Readings where the pages are silent or differ:
  * A block's hash covers its parent block's hash and its own token ids
    (chained), so only a true prefix matches: K/V at a position depend on
    every earlier token.  Matching stops at the first miss.  The hash is
    64-bit FNV-1a over the parent hash (8 bytes, little-endian) followed by the
    block's token ids (4 bytes each, little-endian); the parent of block 0 is
    0.  A hit also compares the stored token ids.
  * Only full blocks of a prompt are registered, when the sequence is
    created, so a cached block is never written (no copy-on-write for it).
    By default a block leaves the map when its refcount reaches 0.
  * Eviction ([PidokuInfra 10] section 10 A names it beside the prefix hash
    table, without rules), when retention is switched on: a registered block
    whose refcount reaches 0 stays registered as evictable, in order of
    release, the blocks one call frees from the last to the first (matching
    stops at a prompt's first miss, so a prompt should lose its tail before
    its head); a prompt that hits it takes it back; an allocation uses the free
    stack and, when that is short, moves the least recently released
    evictable blocks onto it one at a time (dropping their hash entries)
    before taking the top n.  Evictable blocks count as free.  Switching
    retention off frees the evictable blocks, oldest first.
  * The free order is a parameter (the stack's bottom first).  The default is
    the Go constructor's: ids pushed from num_blocks-1 down to 0.
  * A failed append (no free block for a new block or for a copy) changes no
    state.  (The Go AppendToken bumps the length before allocating; the
    nano-vLLM allocate() and the Go Allocate() change nothing on failure, and
    that convention is taken for every call.)
  * Copy-on-write: with refcount n on the written block, each of the first
    n-1 writers copies, and the last one writes in place.
"""


FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3


def fnv1a64(data):
    """64-bit FNV-1a of a byte string (offset basis, then xor-multiply per byte)."""
    h = FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & 0xFFFFFFFFFFFFFFFF
    return h


def fnv1a64_block(parent, tokens):
    """Hash of one full block: FNV-1a over the parent hash (8 bytes LE) then
    each token id (4 bytes LE)."""
    data = int(parent).to_bytes(8, "little") + b"".join(int(t & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class OracleBlockManager:
    """Free list, refcounts, block tables and copy-on-write, in plain Python."""

    def __init__(self, num_blocks, block_size, free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool shape")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if free_order is None:
            self.free = list(range(num_blocks - 1, -1, -1))
        else:
            self.free = [int(b) for b in free_order]
            if sorted(self.free) != list(range(num_blocks)):
                raise ValueError("free_order must be a permutation of the pool's block ids")
        self.ref = {}
        self.tables = {}
        self.lens = {}
        self._next_seq = 0
        self.cached = {}      # hash -> block (full prompt blocks)
        self.block_key = {}   # block -> (hash, token ids) while registered
        self.hits = 0
        self.lookups = 0
        self.retain = False
        self.evictable = []   # registered blocks at refcount 0, oldest release first

    def _unregister(self, b):
        del self.cached[self.block_key.pop(b)[0]]

    def set_retention(self, on):
        if not on:
            for b in self.evictable:
                self._unregister(b)
                self.free.append(b)
            self.evictable = []
        self.retain = bool(on)

    # ---- block-level calls (PidokuInfra section 4) ----
    def blocks_needed(self, tokens):
        return (tokens + self.block_size - 1) // self.block_size

    def allocate(self, n):
        """Top n free ids in slice order, refcount 1; None (no change) when short.
        With too few free ids, evictable blocks are evicted onto the stack first."""
        if len(self.free) + len(self.evictable) < n:
            return None
        if n == 0:
            return []
        while len(self.free) < n:
            b = self.evictable.pop(0)
            self._unregister(b)
            self.free.append(b)
        blocks = self.free[len(self.free) - n:]
        del self.free[len(self.free) - n:]
        for b in blocks:
            self.ref[b] = 1
        return list(blocks)

    def free_blocks(self, blocks):
        retained = []
        for b in blocks:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                del self.ref[b]
                if self.retain and b in self.block_key:
                    retained.append(b)
                else:
                    self.free.append(b)
                    if b in self.block_key:
                        self._unregister(b)
        self.evictable.extend(reversed(retained))

    def fork_blocks(self, blocks):
        for b in blocks:
            self.ref[b] += 1
        return list(blocks)

    # ---- sequence-level calls ----
    def new_sequence(self, prompt_len):
        blocks = self.allocate(self.blocks_needed(prompt_len))
        if blocks is None:
            return None
        seq = self._next_seq
        self._next_seq += 1
        self.tables[seq] = blocks
        self.lens[seq] = int(prompt_len)
        return seq

    def new_sequence_cached(self, token_ids):
        """Create a sequence for a prompt, reusing cached full blocks of its
        prefix.  Returns (seq, cached_tokens) or None (no state change)."""
        tokens = [int(t) for t in token_ids]
        B = self.block_size
        n_full = len(tokens) // B
        hashes, parent = [], 0
        for j in range(n_full):
            parent = fnv1a64_block(parent, tokens[j * B:(j + 1) * B])
            hashes.append(parent)
        reused, lookups = [], 0
        for j in range(n_full):
            lookups += 1
            b = self.cached.get(hashes[j])
            if b is None or self.block_key[b][1] != tuple(tokens[j * B:(j + 1) * B]):
                break
            reused.append(b)
        need = self.blocks_needed(len(tokens)) - len(reused)
        revived = [b for b in reused if b in self.evictable]
        if len(self.free) + len(self.evictable) - len(revived) < need:
            return None
        for b in revived:
            self.evictable.remove(b)
        for b in reused:
            self.ref[b] = self.ref.get(b, 0) + 1
        fresh = self.allocate(need)
        self.lookups += lookups
        self.hits += len(reused)
        table = reused + fresh
        for j in range(len(reused), n_full):
            b = table[j]
            self.cached[hashes[j]] = b
            self.block_key[b] = (hashes[j], tuple(tokens[j * B:(j + 1) * B]))
        seq = self._next_seq
        self._next_seq += 1
        self.tables[seq] = table
        self.lens[seq] = len(tokens)
        return seq, len(reused) * B

    def append_token(self, seq):
        """Make room for the next token of ``seq``.

        Returns (slot, cow_pair) where cow_pair is (src, dst) or None, or None
        when the pool has no block to give (no state change)."""
        table = self.tables[seq]
        pos = self.lens[seq]
        logical = pos // self.block_size
        pair = None
        if pos % self.block_size == 0:
            got = self.allocate(1)
            if got is None:
                return None
            table.append(got[0])
        else:
            old = table[logical]
            if self.ref[old] > 1:
                got = self.allocate(1)
                if got is None:
                    return None
                self.ref[old] -= 1
                table[logical] = got[0]
                pair = (old, got[0])
        self.lens[seq] = pos + 1
        return self.physical_index(seq, pos), pair

    def fork(self, parent):
        child = self._next_seq
        self._next_seq += 1
        self.tables[child] = self.fork_blocks(self.tables[parent])
        self.lens[child] = self.lens[parent]
        return child

    def free_seq(self, seq):
        if seq not in self.tables:
            raise KeyError("unknown or already freed sequence %r" % (seq,))
        self.free_blocks(self.tables.pop(seq))
        del self.lens[seq]

    def physical_index(self, seq, pos):
        table = self.tables[seq]
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def stats(self):
        """(free, used, shared) block counts."""
        shared = sum(1 for r in self.ref.values() if r > 1)
        free = len(self.free) + len(self.evictable)
        return free, self.num_blocks - free, shared


def run_script(num_blocks, block_size, free_order, script, manager=None):
    """Run a workload's block-manager script: ("new", tokens), ("new_cached",
    token_ids), ("fork", parent), ("free", seq), ("append", seq, count),
    ("retain", on), on a fresh manager or on ``manager``.  Sequences are numbered in creation order.

    Returns a dict with the manager, the final ``tables`` (list per sequence),
    ``lens``, the ``slots`` of every appended token in script order, the
    copy-on-write ``pairs`` in the order they were made, and
    ``written_refcounts``: the refcount of each written block at write time."""
    import numpy as np

    m = manager if manager is not None else OracleBlockManager(num_blocks, block_size, free_order)
    slots, pairs, written_refs = [], [], []
    for op in script:
        if op[0] == "new":
            if m.new_sequence(op[1]) is None:
                raise RuntimeError("pool exhausted creating a sequence")
        elif op[0] == "new_cached":
            got = m.new_sequence_cached(op[1])
            if got is None:
                raise RuntimeError("pool exhausted creating a sequence")
            seq, cached = got
            # every prompt position has a K/V row; cached ones are not written
            for pos in range(len(op[1])):
                slots.append(-1 if pos < cached else m.physical_index(seq, pos))
                if pos >= cached:
                    written_refs.append(m.ref[m.tables[seq][pos // block_size]])
        elif op[0] == "fork":
            m.fork(op[1])
        elif op[0] == "free":
            m.free_seq(op[1])
        elif op[0] == "retain":
            m.set_retention(op[1])
        elif op[0] == "append":
            for _ in range(op[2]):
                got = m.append_token(op[1])
                if got is None:
                    raise RuntimeError("pool exhausted appending a token")
                slot, pair = got
                slots.append(slot)
                written_refs.append(m.ref[slot // block_size])
                if pair is not None:
                    pairs.append(pair)
        else:
            raise ValueError("unknown op %r" % (op,))
    order = sorted(m.tables)
    return {
        "manager": m,
        "tables": [list(m.tables[s]) for s in order],
        "lens": np.asarray([m.lens[s] for s in order], dtype=np.int32),
        "slots": np.asarray(slots, dtype=np.int64),
        "pairs": np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
        "written_refcounts": written_refs,
    }



def sampling_memory(prompt_len, gen_lens, block_size):
    """Parallel sampling with and without sharing ([PidokuInfra 10] section
    10 E, on the sharing of section 5): blocks held after every sample has
    generated its tokens, when the samples fork one prompt sequence (each
    appending in turn) and when each holds its own prompt.  Returns
    (shared_blocks, unshared_blocks, copies)."""
    n = len(gen_lens)
    pool = sum(-(-(prompt_len + g) // block_size) for g in gen_lens) + 1
    m = OracleBlockManager(pool, block_size)
    root = m.new_sequence(prompt_len)
    seqs = [root] + [m.fork(root) for _ in range(n - 1)]
    copies = 0
    for seq, g in zip(seqs, gen_lens):
        for _ in range(g):
            copies += m.append_token(seq)[1] is not None
    u = OracleBlockManager(pool, block_size)
    for g in gen_lens:
        seq = u.new_sequence(prompt_len)
        for _ in range(g):
            u.append_token(seq)
    return m.stats()[1], u.stats()[1], copies

def pad_tables(tables, max_blocks):
    """Tables as an int32 [num_seqs, max_blocks] array, unused entries -1."""
    import numpy as np

    out = np.full((len(tables), max(1, max_blocks)), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out
