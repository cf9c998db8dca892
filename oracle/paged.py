"""Page allocator of a paged KV cache, written out plainly (test infrastructure).

The self-speculative decoding page (m.lqnn.cn/news/278124) asks in §3.3 that
a rollback be page-granular -- after a verification round the cache keeps
exactly the accepted prefix, so a sequence gives back whole pages past its
committed length and its write pointer equals its length -- and in §4.5 that
sequences of a batch keep their own offsets.  The pages leave the method's
arithmetic unchanged; what they add is bookkeeping: which physical page holds
which block of a sequence's slots.  This module states that bookkeeping in
the simplest form that makes it reproducible, so the CUDA path's page tables
can be compared with it entry for entry:

* the pool is a stack of free page ids; at creation it is ordered so that the
  first page taken is page 0, then 1, 2, ...;
* ``ensure(ends)``: before a call writes slots, walking the sequences in
  order, every block ``p`` of sequence ``b`` with ``p * page < ends[b]`` that
  has no page takes the top of the stack (blocks in increasing order); an
  empty stack is a capacity error and stops that sequence's walk;
* ``release(lengths)``: after a commit or a change of lengths, walking the
  sequences in order, every block at or past ``ceil(length / page)`` that
  holds a page pushes it back, blocks in decreasing order.

Slot ``s`` of sequence ``b`` lives in page ``table[b][s // page]`` at row
``s % page``.  Only this module and the tests use it; nothing here is shared
with the CUDA path.
"""
from __future__ import annotations


class PoolExhausted(Exception):
    """An ``ensure`` needed more pages than the pool had free."""


class PagePool:
    """Page tables of ``batch`` sequences over a pool of ``n_pages`` pages."""

    def __init__(self, batch, max_ctx, page, n_pages):
        if page < 1 or n_pages < 1 or batch < 1 or max_ctx < 1:
            raise ValueError("bad pool sizes")
        self.batch, self.max_ctx, self.page, self.n_pages = batch, max_ctx, page, n_pages
        self.max_pages = -(-max_ctx // page)
        self.table = [[-1] * self.max_pages for _ in range(batch)]
        # the top of the stack is the end of the list: page 0 is taken first
        self.free = list(range(n_pages - 1, -1, -1))

    def blocks(self, n_slots):
        """Blocks of ``page`` slots that cover the first ``n_slots`` slots."""
        return -(-int(n_slots) // self.page)

    def ensure(self, ends):
        """Give every block below ``ends[b]`` of sequences ``b = 0, 1, ...`` a page.

        ``ends`` may be shorter than the batch (the later sequences need
        nothing).  Raises :class:`PoolExhausted` after handing out every page
        it could, in order, when the stack runs empty; a sequence whose end is
        past ``max_ctx`` raises ``ValueError`` after its first ``max_pages``
        blocks are served.
        """
        short = False
        beyond = False
        for b, end in enumerate(ends):
            need = self.blocks(end)
            if need > self.max_pages:
                beyond = True
                need = self.max_pages
            for p in range(need):
                if self.table[b][p] >= 0:
                    continue
                if not self.free:
                    short = True
                    break
                self.table[b][p] = self.free.pop()
        if beyond:
            raise ValueError("a sequence addresses slots past max_ctx")
        if short:
            raise PoolExhausted("page pool exhausted")

    def ensure_relative(self, lengths, n_new):
        """``ensure`` for calls that append ``n_new[b]`` slots after ``lengths[b]``."""
        self.ensure([int(l) + int(n) for l, n in zip(lengths, n_new)])

    def release(self, lengths):
        """Return the pages of every block at or past ``ceil(lengths[b] / page)``."""
        for b, n in enumerate(lengths):
            keep = self.blocks(n)
            for p in range(self.max_pages - 1, keep - 1, -1):
                if self.table[b][p] >= 0:
                    self.free.append(self.table[b][p])
                    self.table[b][p] = -1

    def set_lengths(self, lengths):
        """What a change of committed lengths does: release past them, then cover them."""
        self.release(lengths)
        self.ensure(lengths)

    def locate(self, b, s):
        """(page, row in page) of slot ``s`` of sequence ``b``; the page is -1 if none is held."""
        return self.table[b][s // self.page], s % self.page

    def free_count(self):
        return len(self.free)
