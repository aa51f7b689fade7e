"""Reference prefix cache by chained block hashes, in plain Python.

TEST INFRASTRUCTURE (see the package docstring).

Prefix caching by block hashes ("Paged Attention: Managing the KV Cache Like
Virtual Memory", inference-serving tag page); blocks chained by hashes, so that
one character changed early in a system prompt voids the cached blocks after
it (the posts on the pagedattention tag, on vLLM's prompt caching).  A full
block is found again by the hash of its tokens chained to the hash of the
block before it, so a block is reused only when the whole prefix up to and
including it is the same.

The pages fix neither the hash nor the eviction rule; the readings taken
(the library's host allocator must reproduce them bit for bit):
  * h_k = FNV-1a 64-bit over the 8 little-endian bytes of h_{k-1} followed by
    the block's 16 token ids as 4-byte little-endian two's-complement
    integers; h_{-1} = 0.  FNV-1a: start at 14695981039346656037, for each
    byte xor it in, then multiply by 1099511628211 modulo 2**64.
  * Only full blocks are hashed, when their last token is appended with its
    id (append_token); a sequence that ever appends without an id
    (append_slot) stops being hashed.  A hash already in the index keeps its
    older block.
  * The index stores, per hash, the block, the parent hash and the 16 token
    ids; a lookup accepts an entry only if all of them match (a hash collision
    is a miss).
  * A freed block whose count reaches 0 joins the back of the FIFO free list
    but keeps its index entry; a lookup that hits it takes it back out of the
    free list.  Allocation takes the front block and drops its index entry.
  * seq_add_cached(seq, tokens) walks the prompt's full blocks from the start
    and shares every block found, stopping at the first miss; the sequence
    then holds 16 x hits tokens and the caller appends the rest.
Everything else (FIFO order, copy-on-write, fork, OOM) is the reference
allocator's policy.
"""
FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1


def fnv1a64(data, h=FNV_OFFSET):
    for b in bytes(data):
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent, tokens):
    data = int(parent).to_bytes(8, "little") + b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
    return fnv1a64(data)


class PrefixCacheAllocator:
    def __init__(self, num_blocks, block_size=16, free_order=None):
        self.num_blocks = num_blocks
        self.bs = block_size
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free_order must be a permutation"
        self.free = list(order)
        self.refcount = [0] * num_blocks
        self.tables, self.lengths = {}, {}
        self.tokens = {}    # seq -> token ids appended with ids (None once untracked)
        self.chain = {}     # seq -> hashes of its full blocks
        self.index = {}     # hash -> (block, parent hash, tokens)
        self.key_of = {}    # block -> hash while indexed
        self.queries = 0
        self.hits = 0

    # -- blocks
    def _take(self):
        if not self.free:
            raise MemoryError("no free block")
        b = self.free.pop(0)
        if b in self.key_of:
            del self.index[self.key_of.pop(b)]
        self.refcount[b] = 1
        return b

    def _share(self, b):
        if self.refcount[b] == 0:
            self.free.remove(b)
        self.refcount[b] += 1

    # -- sequences
    def seq_add(self, seq):
        if seq < 0 or seq in self.tables:
            raise ValueError("bad or duplicate sequence id")
        self.tables[seq], self.lengths[seq] = [], 0
        self.tokens[seq], self.chain[seq] = [], []

    def seq_add_cached(self, seq, prompt):
        self.seq_add(seq)
        parent = 0
        for k in range(len(prompt) // self.bs):
            toks = tuple(int(t) for t in prompt[k * self.bs:(k + 1) * self.bs])
            h = block_hash(parent, toks)
            self.queries += 1
            e = self.index.get(h)
            if e is None or e[1] != parent or e[2] != toks:
                break
            self.hits += 1
            self._share(e[0])
            self.tables[seq].append(e[0])
            self.tokens[seq].extend(toks)
            self.chain[seq].append(h)
            self.lengths[seq] += self.bs
            parent = h
        return self.lengths[seq]

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables or child < 0:
            raise ValueError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        self.tokens[child] = None if self.tokens[parent] is None else list(self.tokens[parent])
        self.chain[child] = list(self.chain[parent])
        for b in self.tables[child]:
            self.refcount[b] += 1

    def _append(self, seq):
        table, pos, bs = self.tables[seq], self.lengths[seq], self.bs
        cow = (-1, -1)
        if pos % bs == 0:
            table.append(self._take())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                b = self._take()
                self.refcount[last] -= 1
                table[-1] = b
                cow = (last, b)
        self.lengths[seq] = pos + 1
        return table[pos // bs] * bs + pos % bs, cow[0], cow[1]

    def append_slot(self, seq):
        r = self._append(seq)
        self.tokens[seq] = None
        return r

    def append_token(self, seq, token):
        r = self._append(seq)
        toks = self.tokens[seq]
        if toks is not None:
            toks.append(int(token))
            n = len(toks)
            if n % self.bs == 0:
                k = n // self.bs - 1
                parent = self.chain[seq][k - 1] if k > 0 else 0
                block_toks = tuple(toks[k * self.bs:])
                h = block_hash(parent, block_toks)
                self.chain[seq].append(h)
                b = self.tables[seq][k]
                if h not in self.index and b not in self.key_of:
                    self.index[h] = (b, parent, block_toks)
                    self.key_of[b] = h
        return r

    def seq_free(self, seq):
        for b in self.tables.pop(seq):
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.lengths[seq], self.tokens[seq], self.chain[seq]

    def table(self, seq):
        return list(self.tables[seq])

    def block_key(self, b):
        return self.key_of.get(b)
