"""Reference KV block manager (oracle, test infrastructure only).

A direct restatement of the block manager the pages describe:

* MiniPaged-Qwen §8.1 (SequenceState: id, length, block table), §8.2 (the
  fixed pool and its free list), §9 (append_token), §5.3 (release walks the
  table and returns every block), §15 (invariants).
* mini-vLLM Block Manager, sections "prefill 时如何分配 block" (prefill takes
  ceil(n / block_size) blocks from the free list at once), "decode 时如何追加
  slot" (a new block only when the write position starts a new logical
  block), "释放 block" (release exactly once), "正确性不变量" (invariants and
  the debug owner table).
* LLM-algo ch.22, Step 4 reference answer: prefill is all-or-nothing on
  OOM, a decode that needs a block but finds none leaves the length and the
  table unchanged, a second prefill of a live request is rejected, request
  ids are non-negative and prompt lengths positive.

Readings where the pages are silent or disagree (each listed in the design
notes):

* Free-list order: blocks are taken from the FRONT of the free list and
  released blocks are appended at the BACK in block-table order, with no
  sort.  The mini-vLLM lifecycle example (free [3, 8, 1, 5, 7, ...] ->
  table [3, 8, 1], free [5, 7, ...]) and the LLM-algo answer
  (``free_blocks[:needed]``, ``pop(0)``) take from the front.  The LLM-algo
  answer sorts the free list on release; we do not, so seeded initial orders
  and churn survive -- its release test is checked as set equality.
* Boundary test: allocate iff ``length // block_size == len(table)``
  (MiniPaged-Qwen §9), which agrees with LLM-algo's ``new_len % bs == 1`` for
  block sizes >= 2.
* A released id may be prefilled again; releasing an id twice without a new
  prefill in between is a double free; releasing an id never seen is an
  unknown sequence.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Iterable, List, Optional, Sequence


class OracleError(Exception):
    """An error the manager reports; ``code`` names the condition."""

    def __init__(self, code: str, msg: str = ""):
        super().__init__(f"{code}: {msg}" if msg else code)
        self.code = code


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class SequenceState:
    """MiniPaged-Qwen §8.1: one live sequence's metadata."""

    sequence_id: int
    sequence_length: int = 0  # tokens written == next append position
    block_table: List[int] = field(default_factory=list)


class BlockManager:
    """Reference manager over a fixed pool of ``num_blocks`` physical blocks."""

    def __init__(self, num_blocks: int, block_size: int,
                 initial_free_order: Optional[Sequence[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise OracleError("INVALID_ARG", "num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        if initial_free_order is None:
            order = list(range(self.num_blocks))
        else:
            order = [int(x) for x in initial_free_order]
            if sorted(order) != list(range(self.num_blocks)):
                raise OracleError("INVALID_ARG", "initial free order must be a permutation of the pool")
        self.free_blocks: List[int] = order
        self.sequences: Dict[int, SequenceState] = {}
        self.released_ids: set = set()

    # -- allocation primitives -------------------------------------------------
    def _take_front(self, count: int) -> List[int]:
        taken = self.free_blocks[:count]
        del self.free_blocks[:count]
        return taken

    @staticmethod
    def _slot(table: List[int], pos: int, bs: int) -> int:
        """MiniPaged-Qwen §3: logical block = pos // bs, offset = pos % bs,
        physical block = table[logical block], slot = physical * bs + offset."""
        return table[pos // bs] * bs + pos % bs

    # -- admission checks (mini-vLLM Block Manager, scheduler interplay) -------
    def can_allocate(self, num_tokens: int) -> bool:
        if num_tokens <= 0:
            raise OracleError("INVALID_ARG", "num_tokens must be positive")
        return _ceil_div(num_tokens, self.block_size) <= len(self.free_blocks)

    def can_append_slots(self, seq_ids: Iterable[int]) -> bool:
        need = 0
        for sid in seq_ids:
            st = self._get(sid)
            if st.sequence_length // self.block_size == len(st.block_table):
                need += 1
        return need <= len(self.free_blocks)

    # -- prefill ---------------------------------------------------------------
    def allocate_for_prefill(self, seq_id: int, num_tokens: int) -> List[int]:
        """Allocate ceil(n / bs) blocks at once and return the n prompt slots.

        All or nothing: on OOM neither the free list nor any table changes
        (LLM-algo ch.22 Step 4, TODO 2 and its analysis)."""
        if seq_id < 0 or num_tokens <= 0:
            raise OracleError("INVALID_ARG", "seq_id must be >= 0 and num_tokens > 0")
        if seq_id in self.sequences:
            raise OracleError("DUPLICATE_SEQ", f"sequence {seq_id} already prefilled")
        need = _ceil_div(num_tokens, self.block_size)
        if need > len(self.free_blocks):
            raise OracleError("OOM", f"need {need} blocks, {len(self.free_blocks)} free")
        st = SequenceState(seq_id, num_tokens, self._take_front(need))
        self.sequences[seq_id] = st
        self.released_ids.discard(seq_id)
        return [self._slot(st.block_table, t, self.block_size) for t in range(num_tokens)]

    # -- decode ----------------------------------------------------------------
    def append_slot_for_decode(self, seq_id: int) -> int:
        """MiniPaged-Qwen §9 append_token: slot for position L, allocating a
        block only when L starts a new logical block; then L += 1.  On OOM the
        sequence is unchanged (LLM-algo ch.22, decode rollback test)."""
        st = self._get(seq_id)
        bs = self.block_size
        L = st.sequence_length
        if L // bs == len(st.block_table):
            if not self.free_blocks:
                raise OracleError("OOM", "no free block for decode append")
            st.block_table.append(self._take_front(1)[0])
        slot = self._slot(st.block_table, L, bs)
        st.sequence_length = L + 1
        return slot

    def append_slots(self, seq_id: int, num_tokens: int) -> List[int]:
        """``num_tokens`` consecutive decode appends, all or nothing on OOM."""
        if num_tokens <= 0:
            raise OracleError("INVALID_ARG", "num_tokens must be positive")
        st = self._get(seq_id)
        need = _ceil_div(st.sequence_length + num_tokens, self.block_size) - len(st.block_table)
        if need > len(self.free_blocks):
            raise OracleError("OOM", f"need {need} blocks, {len(self.free_blocks)} free")
        return [self.append_slot_for_decode(seq_id) for _ in range(num_tokens)]

    def decode_step(self, seq_ids: Sequence[int]) -> List[int]:
        """One decode token for each listed sequence, all or nothing on OOM."""
        ids = [int(s) for s in seq_ids]
        if len(set(ids)) != len(ids):
            raise OracleError("INVALID_ARG", "a sequence appears twice in one decode step")
        for sid in ids:
            self._get(sid)
        if not self.can_append_slots(ids):
            raise OracleError("OOM", "not enough free blocks for this decode step")
        return [self.append_slot_for_decode(sid) for sid in ids]

    # -- release ---------------------------------------------------------------
    def free_sequence(self, seq_id: int) -> None:
        """MiniPaged-Qwen §5.3 / mini-vLLM "释放 block": return every block once.

        The table is validated first (LLM-algo ch.22 release checks: no
        duplicates, in range, none already free); a corrupt table is an
        invariant violation and nothing is changed."""
        if seq_id not in self.sequences:
            if seq_id in self.released_ids:
                raise OracleError("DOUBLE_FREE", f"sequence {seq_id} already released")
            raise OracleError("UNKNOWN_SEQ", f"sequence {seq_id} is not live")
        table = self.sequences[seq_id].block_table
        if len(set(table)) != len(table):
            raise OracleError("INVARIANT", "duplicate block in table")
        if any(b < 0 or b >= self.num_blocks for b in table):
            raise OracleError("INVARIANT", "block index out of range")
        free_set = set(self.free_blocks)
        if any(b in free_set for b in table):
            raise OracleError("INVARIANT", "table holds a free block")
        self.free_blocks.extend(table)
        del self.sequences[seq_id]
        self.released_ids.add(seq_id)

    # -- metadata export (MiniPaged-Qwen §16.2 get_block_table_tensor, get_seq_lens_tensor)
    def export(self, seq_ids: Sequence[int], max_blocks: int):
        """Return (block_tables [n][max_blocks] padded with -1, seq_lens [n])."""
        tables, lens = [], []
        for sid in seq_ids:
            st = self._get(sid)
            if len(st.block_table) > max_blocks:
                raise OracleError("INVALID_ARG", "max_blocks smaller than a table")
            tables.append(st.block_table + [-1] * (max_blocks - len(st.block_table)))
            lens.append(st.sequence_length)
        return tables, lens

    def block_table(self, seq_id: int) -> List[int]:
        return list(self._get(seq_id).block_table)

    def seq_len(self, seq_id: int) -> int:
        return self._get(seq_id).sequence_length

    def num_free_blocks(self) -> int:
        return len(self.free_blocks)

    # -- invariants (MiniPaged-Qwen §15; mini-vLLM "正确性不变量"; LLM-algo Step 3 table)
    def invariants_ok(self) -> bool:
        bs = self.block_size
        allocated: List[int] = []
        owner: Dict[int, int] = {}
        for sid, st in self.sequences.items():
            if len(st.block_table) != _ceil_div(st.sequence_length, bs):
                return False  # length must match the tail block
            for b in st.block_table:
                if b < 0 or b >= self.num_blocks:
                    return False  # invalid physical index
                if b in owner:
                    return False  # one block, two owners
                owner[b] = sid
            allocated.extend(st.block_table)
        free = self.free_blocks
        if len(set(free)) != len(free):
            return False
        if any(b < 0 or b >= self.num_blocks for b in free):
            return False
        if set(allocated) & set(free):
            return False
        return len(allocated) + len(free) == self.num_blocks

    def _get(self, seq_id: int) -> SequenceState:
        if seq_id not in self.sequences:
            raise OracleError("UNKNOWN_SEQ", f"sequence {seq_id} is not live")
        return self.sequences[seq_id]
