"""Plain-Python oracle of the host block manager (TEST INFRASTRUCTURE ONLY).

Only ``tests/`` may import this module; the library never does, and this
module shares no code with it.  It restates, with lists, dicts and tuples,
the bookkeeping of a paged KV cache ("03 - Engines Papers", section 2
PagedAttention (vLLM): block table, refcounts, copy on write; section 4
SGLang (RadixAttention): prefix reuse with LRU eviction; "The LLM inference
engine playbook", Theme 3) under the deterministic policy that
``include/pa_block_manager.h`` states:

  * free blocks: a FIFO queue starting 0..N-1; allocation takes its head;
    with the queue empty, the least recently released cached block with no
    holder is evicted and taken;
  * a sequence's blocks are released last block first; a block whose
    refcount reaches 0 is parked until the step ends, then joins the free
    queue (uncached) or the eviction order (cached), in parking order;
  * the prefix cache maps the exact token prefix that ends a full block to
    that block (here a tuple key, so no hashing is involved); a block is
    registered when it becomes full if the sequence's previous block is
    registered (or it is the first block) and no block holds that prefix;
  * evicting a cached block drops every cached prefix that extends its own;
    those blocks that nobody holds leave the eviction order for the free
    queue's tail in ascending id;
  * admission reuses the longest run of cached prefixes of the prompt, at
    most floor((n - 1) / B) blocks;
  * appending into a shared partial block copies it to a new block first
    (a copy pair of the step), unless the block already got a slot in this
    step (then the call is refused with STEP);
  * every call checks first and changes nothing when it fails.
"""
from __future__ import annotations

from collections import deque

OK, INVALID, NO_BLOCKS, STEP = 0, -1, -6, -7


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self.N, self.B, self.caching = num_blocks, block_size, prefix_caching
        self.ref = [0] * num_blocks
        self.free = deque(range(num_blocks))
        self.seqs = {}            # id -> {"blocks": [...], "tokens": [...]}
        self.copies = []          # this step's (src, dst)
        self.step = 1
        self.written = [0] * num_blocks
        self.parked = []          # blocks parked in this step, in parking order
        self.cache = {}           # prefix tuple -> block
        self.prefix_of = {}       # block -> prefix tuple (registered blocks)
        self.lru = []             # evictable cached blocks, least recently released first

    # ------------------------------------------------------------ helpers
    def available(self) -> int:
        return len(self.free) + len(self.lru)

    def _evict(self, b: int) -> None:
        self.lru.remove(b)
        mine = self.prefix_of[b]
        dropped = []
        for key, c in list(self.cache.items()):
            if len(key) > len(mine) and key[:len(mine)] == mine:
                dropped.append(c)
        for c in dropped + [b]:
            del self.cache[self.prefix_of[c]]
            del self.prefix_of[c]
        for c in sorted(dropped):
            if c in self.lru:
                self.lru.remove(c)
                self.free.append(c)

    def _alloc(self) -> int:
        if self.free:
            b = self.free.popleft()
        else:
            b = self.lru[0]
            self._evict(b)
        self.ref[b] = 1
        return b

    def _acquire(self, b: int) -> None:
        if self.ref[b] == 0:
            if b in self.lru:
                self.lru.remove(b)
            elif b in self.parked:
                self.parked.remove(b)
        self.ref[b] += 1

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.parked.append(b)

    def _register(self, blocks, tokens, j: int) -> None:
        if not self.caching:
            return
        b = blocks[j]
        if b in self.prefix_of:
            return
        if j > 0 and blocks[j - 1] not in self.prefix_of:
            return
        key = tuple(tokens[:(j + 1) * self.B])
        if key in self.cache:
            return
        self.cache[key] = b
        self.prefix_of[b] = key

    # ------------------------------------------------------------ API
    def add_sequence(self, seq_id, tokens):
        """Returns (status, slots list, num_cached)."""
        n, B = len(tokens), self.B
        if n < 1 or seq_id in self.seqs:
            return INVALID, None, 0
        hit = []
        if self.caching:
            for j in range((n - 1) // B):
                b = self.cache.get(tuple(tokens[:(j + 1) * B]))
                if b is None:
                    break
                hit.append(b)
        need = -(-n // B)
        if self.available() - sum(1 for b in hit if b in self.lru) < need - len(hit):
            return NO_BLOCKS, None, 0
        blocks = []
        for b in hit:
            self._acquire(b)
            blocks.append(b)
        for _ in range(need - len(hit)):
            b = self._alloc()
            self.written[b] = self.step
            blocks.append(b)
        cached = len(hit) * B
        slots = [-1 if p < cached else blocks[p // B] * B + p % B for p in range(n)]
        tokens = list(tokens)
        for j in range(len(hit), n // B):
            self._register(blocks, tokens, j)
        self.seqs[seq_id] = {"blocks": blocks, "tokens": tokens}
        return OK, slots, cached

    def append_token(self, seq_id, token):
        """Returns (status, slot)."""
        if seq_id not in self.seqs:
            return INVALID, None
        s, B = self.seqs[seq_id], self.B
        p = len(s["tokens"])
        j = p // B
        new_block = p % B == 0
        cow = not new_block and self.ref[s["blocks"][j]] > 1
        if cow and self.written[s["blocks"][j]] == self.step:
            return STEP, None
        if (new_block or cow) and self.available() < 1:
            return NO_BLOCKS, None
        if new_block:
            s["blocks"].append(self._alloc())
        elif cow:
            old = s["blocks"][j]
            new = self._alloc()
            self.copies.append((old, new))
            self._release(old)
            s["blocks"][j] = new
        s["tokens"].append(token)
        self.written[s["blocks"][j]] = self.step
        if (p + 1) % B == 0:
            self._register(s["blocks"], s["tokens"], j)
        return OK, s["blocks"][j] * B + p % B

    def fork(self, parent_id, child_id):
        if parent_id not in self.seqs or child_id in self.seqs:
            return INVALID
        s = self.seqs[parent_id]
        for b in s["blocks"]:
            self._acquire(b)
        self.seqs[child_id] = {"blocks": list(s["blocks"]), "tokens": list(s["tokens"])}
        return OK

    def free_sequence(self, seq_id):
        if seq_id not in self.seqs:
            return INVALID
        for b in reversed(self.seqs.pop(seq_id)["blocks"]):
            self._release(b)
        return OK

    def end_step(self):
        """Returns the step's copy pairs."""
        pairs = list(self.copies)
        self.copies = []
        for b in self.parked:
            if b in self.prefix_of:
                self.lru.append(b)
            else:
                self.free.append(b)
        self.parked = []
        self.step += 1
        return pairs

    def build_tables(self, seq_ids, max_blocks):
        """Returns (status, tables rows, seq_lens)."""
        rows, lens = [], []
        for i in seq_ids:
            if i not in self.seqs or len(self.seqs[i]["blocks"]) > max_blocks:
                return INVALID, None, None
            b = self.seqs[i]["blocks"]
            rows.append(b + [-1] * (max_blocks - len(b)))
            lens.append(len(self.seqs[i]["tokens"]))
        return OK, rows, lens

    def counters(self):
        """(free, parked, cached, evictable)."""
        return len(self.free), len(self.parked), len(self.cache), len(self.lru)
