"""Host bookkeeping for a paged KV pool.

A pool of ``num_blocks`` physical blocks of ``block_size`` token slots each.
Every sequence owns a block table (logical block -> physical block). Blocks
are reference counted so that sequences can share them; a write into a shared,
partly filled block first copies it (copy-on-write). With prefix caching on,
every full block gets a key chained from its parent's key, its token ids and,
for the first block, a per-request salt; a new prompt reuses the unbroken run
of cached full blocks from its start. Released blocks go to the tail of a
least-recently-used free queue and keep their key until the block is handed
out again.

Behaviour follows "Batching and the KV Cache" (Chapter 2, the block-manager
teaching model and its demo: block tables, reference counts, copy-on-write,
fork, hash chain with salt, LRU free queue), "MLSys Engineer -- Inference
Systems Q&A" Q1 (at most one partly filled block per sequence; shared blocks
are copied on write) and "Design an LLM Inference API with GPU Batching",
4.2 (free blocks, per-block reference counts, prefix index).

The manager decides where tokens go; it moves no KV data. ``append`` returns
the slot of the new token and, when copy-on-write fired, the (source,
destination) block pair whose contents the caller must copy.
"""
from __future__ import annotations

import hashlib
import struct
from collections import OrderedDict
from dataclasses import dataclass
from typing import Iterable, Optional


class OutOfBlocks(MemoryError):
    """No free block is left: the caller must preempt a sequence."""


@dataclass(frozen=True)
class AppendResult:
    slot: int                                   # block * block_size + offset
    copy_on_write: Optional[tuple[int, int]]    # (src block, dst block) or None


def _chain_key(parent: Optional[bytes], tokens: Iterable[int], salt: str) -> bytes:
    """Key of a full block: sha256 over the parent's key (or the salt, for the
    first block of a sequence) and the block's token ids."""
    h = hashlib.sha256()
    if parent is None:
        h.update(b"root\x00" + salt.encode("utf-8"))
    else:
        h.update(b"next\x00" + parent)
    toks = list(tokens)
    h.update(struct.pack(f"<{len(toks)}q", *toks))
    return h.digest()


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16,
                 free_order: Optional[Iterable[int]] = None,
                 prefix_caching: bool = True):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("num_blocks must be >= 0 and block_size > 0")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.prefix_caching = prefix_caching
        # LRU free queue: the first entry is handed out next.
        self._free: "OrderedDict[int, None]" = OrderedDict((b, None) for b in order)
        self._refs = [0] * num_blocks
        self._tokens: list[list[int]] = [[] for _ in range(num_blocks)]
        self._key: list[Optional[bytes]] = [None] * num_blocks
        self._cached: dict[bytes, int] = {}         # key of a full block -> block id
        self._tables: dict[str, list[int]] = {}
        self._salts: dict[str, str] = {}

    # ---- queries -------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def refcount(self, block: int) -> int:
        return self._refs[block]

    def block_table(self, seq: str) -> list[int]:
        return list(self._tables[seq])

    def num_tokens(self, seq: str) -> int:
        table = self._tables[seq]
        if not table:
            return 0
        return (len(table) - 1) * self.block_size + len(self._tokens[table[-1]])

    def slot(self, seq: str, position: int) -> int:
        """Flat slot of logical token ``position`` of ``seq``."""
        table = self._tables[seq]
        return table[position // self.block_size] * self.block_size + position % self.block_size

    def sequences(self) -> list[str]:
        return list(self._tables)

    # ---- internals -----------------------------------------------------
    def _allocate(self, tokens: list[int]) -> int:
        if not self._free:
            raise OutOfBlocks("out of KV blocks: preempt a sequence")
        block, _ = self._free.popitem(last=False)
        key = self._key[block]
        if key is not None and self._cached.get(key) == block:
            del self._cached[key]          # reuse evicts the prefix the block held
        self._refs[block] = 1
        self._tokens[block] = list(tokens)
        self._key[block] = None
        return block

    def _seal_if_full(self, block: int, parent: Optional[bytes], salt: str) -> None:
        if self.prefix_caching and len(self._tokens[block]) == self.block_size:
            key = _chain_key(parent, self._tokens[block], salt)
            self._key[block] = key
            self._cached.setdefault(key, block)

    def _parent_key(self, table: list[int], index: int) -> Optional[bytes]:
        return self._key[table[index - 1]] if index > 0 else None

    # ---- operations ----------------------------------------------------
    def admit(self, seq: str, prompt: Iterable[int], salt: str = "") -> int:
        """Build the block table of a new sequence; return how many prompt
        tokens were found in the prefix cache (a multiple of block_size)."""
        if seq in self._tables:
            raise KeyError(f"sequence {seq!r} already admitted")
        prompt = [int(t) for t in prompt]
        bs = self.block_size
        table: list[int] = []
        hits = 0
        try:
            for start in range(0, len(prompt), bs):
                chunk = prompt[start:start + bs]
                parent = self._parent_key(table, len(table))
                found = None
                if self.prefix_caching and len(chunk) == bs and hits == start:
                    found = self._cached.get(_chain_key(parent, chunk, salt))
                if found is not None:
                    if self._refs[found] == 0:
                        del self._free[found]
                    self._refs[found] += 1
                    hits += bs
                    table.append(found)
                else:
                    block = self._allocate(chunk)
                    self._seal_if_full(block, parent, salt)
                    table.append(block)
        except OutOfBlocks:
            self._drop(table)
            raise
        self._tables[seq] = table
        self._salts[seq] = salt
        return hits

    def append(self, seq: str, token: int) -> AppendResult:
        """One decode step for ``seq``: place ``token`` in its slot. A full last
        block gets a fresh successor; a shared, partly filled last block is
        first replaced by a private copy (copy-on-write)."""
        table = self._tables[seq]
        salt = self._salts[seq]
        cow = None
        if not table or len(self._tokens[table[-1]]) == self.block_size:
            table.append(self._allocate([]))
        elif self._refs[table[-1]] > 1:
            shared = table[-1]
            private = self._allocate(self._tokens[shared])
            self._refs[shared] -= 1
            table[-1] = private
            cow = (shared, private)
        last = table[-1]
        self._tokens[last].append(int(token))
        self._seal_if_full(last, self._parent_key(table, len(table) - 1), salt)
        return AppendResult(last * self.block_size + len(self._tokens[last]) - 1, cow)

    def fork(self, seq: str, child: str) -> None:
        """The child shares every block of ``seq`` (parallel sampling, beam search)."""
        if child in self._tables:
            raise KeyError(f"sequence {child!r} already admitted")
        table = self._tables[seq]
        for b in table:
            self._refs[b] += 1
        self._tables[child] = list(table)
        self._salts[child] = self._salts[seq]

    def release(self, seq: str) -> None:
        """Drop a finished sequence; blocks whose count reaches zero join the
        free queue's tail, last block first, and stay reusable by key."""
        self._drop(self._tables.pop(seq))
        self._salts.pop(seq, None)

    def _drop(self, table: list[int]) -> None:
        for b in reversed(table):
            self._refs[b] -= 1
            if self._refs[b] == 0:
                self._free[b] = None

    # ---- invariants ----------------------------------------------------
    def wasted_slots(self, seq: str) -> int:
        """Allocated but unused slots of ``seq`` (internal fragmentation)."""
        return len(self._tables[seq]) * self.block_size - self.num_tokens(seq)

    def check(self) -> None:
        """Reference counts equal table occurrences; free blocks have count 0."""
        counts = [0] * self.num_blocks
        for table in self._tables.values():
            for b in table:
                counts[b] += 1
        if counts != self._refs:
            raise AssertionError("reference counts disagree with the block tables")
        for b in self._free:
            if self._refs[b] != 0:
                raise AssertionError(f"block {b} is free with count {self._refs[b]}")
        if len(self._free) + sum(1 for c in counts if c > 0) != self.num_blocks:
            raise AssertionError("blocks leaked: neither free nor referenced")
