"""Plain-Python model of the fixed-block paged K/V allocator (test oracle).

Follows "feat: add paged-attention monolithic decode-only AR foundation"
(lucebox pull 555), Summary: an exact pool of fixed-size blocks, allocation
that is transactional (all or nothing), detection of stale handles, and
release that takes effect immediately.  The pages do not fix an order, so
the policy below is this build's reading, stated exactly so that the C++
allocator can be compared with it handle for handle:

- ids 0 .. n-1; the free list is a stack; a fresh pool pops 0, 1, 2, ...;
- a handle is (generation << 32) | id; generations start at 1 and advance
  by one when the block is released, skipping 0 on wrap-around, so the
  handle value 0 is never valid;
- alloc(n) fails with NOMEM and changes nothing when n exceeds the free
  count; otherwise it pops n ids in stack order;
- free(handles) first validates every handle (id in range, block live,
  generation current, no handle listed twice); any failure returns STALE
  and releases nothing; otherwise blocks are released in list order, each
  pushed on the stack (the last one released is the next one allocated).
"""

OK, NOMEM, STALE, INVALID = 0, -2, -3, -1
MASK32 = 0xFFFFFFFF


class PoolModel:
    def __init__(self, n_blocks: int):
        if n_blocks < 1 or n_blocks > 0x7FFFFFFF:
            raise ValueError("n_blocks out of range")
        self.n = n_blocks
        self.gen = [1] * n_blocks
        self.live = [False] * n_blocks
        self.stack = list(range(n_blocks - 1, -1, -1))  # top of stack = last item

    def free_count(self) -> int:
        return len(self.stack)

    def alloc(self, n: int):
        if n > len(self.stack):
            return NOMEM, []
        out = []
        for _ in range(n):
            i = self.stack.pop()
            self.live[i] = True
            out.append((self.gen[i] << 32) | i)
        return OK, out

    def free(self, handles):
        seen = set()
        for h in handles:
            i, g = h & MASK32, h >> 32
            if i >= self.n or not self.live[i] or self.gen[i] != g or i in seen:
                return STALE
            seen.add(i)
        for h in handles:
            i = h & MASK32
            self.live[i] = False
            g = (self.gen[i] + 1) & MASK32
            self.gen[i] = g if g != 0 else 1
            self.stack.append(i)
        return OK

    @staticmethod
    def block_of(h: int) -> int:
        return h & MASK32
