"""Reference block manager with prefix sharing and copy-on-write (oracle,
test infrastructure only).

Follows "paged-attention-impl-detail" (guijiagi.com), section
Copy-on-Write共享:

* 前缀共享 (share_prefix_blocks): requests with a common prompt prefix hold
  the same ceil(prefix_len / block_size) physical blocks; every extra
  holder adds one to each shared block's ref_count.
* Copy-on-Write机制 (copy_on_write): a request about to modify a block whose
  ref_count is above 1 takes a new block, copies the old block's k and v
  into it, lowers the old block's ref_count by one, gives the new block a
  ref_count of 1 and puts it in its table where the old one was.  With a
  ref_count of 1 the block is its own and is written in place.

"从零实现一个 mini vLLM: Block Manager", section 正确性不变量: a physical block
belongs to one sequence unless prefix caching or copy-on-write is in
place -- the one relaxation made here.

Everything else is ``oracle.block_manager.BlockManager`` unchanged (free
list taken from the front, releases appended at the back in table order,
all-or-nothing allocation).  Readings where the pages leave a step open:

* A child sequence is the parent's first ``prefix_len`` tokens; when
  ``prefix_len`` is not a multiple of the block size, the last shared block
  is only partly the child's, and the first write of either holder into it
  copies it (guijiagi's "needs to modify a shared block").
* A write starts a copy only when it lands in an existing block (position
  L with L % block_size != 0); a write that opens a new logical block takes
  a fresh block as usual.
* A released block returns to the free list when its ref_count reaches 0.
* Copies are reported as (src, dst) block pairs in the order they arose;
  the device applies them before the step's cache writes.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

from .block_manager import BlockManager, OracleError, SequenceState, _ceil_div


class SharingBlockManager(BlockManager):
    """BlockManager plus per-block ref_count, fork and copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int,
                 initial_free_order: Optional[Sequence[int]] = None):
        super().__init__(num_blocks, block_size, initial_free_order)
        self.ref_count: List[int] = [0] * self.num_blocks
        self.copies: List[Tuple[int, int]] = []

    # -- primitives ------------------------------------------------------------
    def _take_front(self, count: int) -> List[int]:
        taken = super()._take_front(count)
        for b in taken:
            self.ref_count[b] = 1
        return taken

    def _needs_copy(self, st: SequenceState) -> bool:
        L = st.sequence_length
        return L % self.block_size != 0 and self.ref_count[st.block_table[-1]] > 1

    def _blocks_for_one_append(self, st: SequenceState) -> int:
        if st.sequence_length // self.block_size == len(st.block_table):
            return 1
        return 1 if self._needs_copy(st) else 0

    # -- sharing ---------------------------------------------------------------
    def fork(self, parent_id: int, child_id: int, prefix_len: int) -> None:
        """share_prefix_blocks for one more request: the child holds the
        parent's first ceil(prefix_len / bs) blocks, each one reference more."""
        parent = self._get(parent_id)
        if child_id < 0:
            raise OracleError("INVALID_ARG", "child id must be >= 0")
        if child_id in self.sequences:
            raise OracleError("DUPLICATE_SEQ", f"sequence {child_id} is live")
        if not 1 <= prefix_len <= parent.sequence_length:
            raise OracleError("INVALID_ARG", "prefix_len outside [1, parent length]")
        n_shared = _ceil_div(prefix_len, self.block_size)
        shared = parent.block_table[:n_shared]
        for b in shared:
            self.ref_count[b] += 1
        self.sequences[child_id] = SequenceState(child_id, prefix_len, list(shared))
        self.released_ids.discard(child_id)

    def take_copies(self) -> List[Tuple[int, int]]:
        out, self.copies = self.copies, []
        return out

    # -- appends (MiniPaged-Qwen §9 with copy_on_write before an in-place write)
    def can_append_slots(self, seq_ids) -> bool:
        need = sum(self._blocks_for_one_append(self._get(sid)) for sid in seq_ids)
        return need <= len(self.free_blocks)

    def append_slot_for_decode(self, seq_id: int) -> int:
        st = self._get(seq_id)
        bs = self.block_size
        L = st.sequence_length
        if L // bs == len(st.block_table):
            if not self.free_blocks:
                raise OracleError("OOM", "no free block for decode append")
            st.block_table.append(self._take_front(1)[0])
        elif self._needs_copy(st):
            if not self.free_blocks:
                raise OracleError("OOM", "no free block for a copy-on-write")
            old = st.block_table[-1]
            new = self._take_front(1)[0]
            self.ref_count[old] -= 1
            st.block_table[-1] = new
            self.copies.append((old, new))
        slot = self._slot(st.block_table, L, bs)
        st.sequence_length = L + 1
        return slot

    def append_slots(self, seq_id: int, num_tokens: int) -> List[int]:
        if num_tokens <= 0:
            raise OracleError("INVALID_ARG", "num_tokens must be positive")
        st = self._get(seq_id)
        need = _ceil_div(st.sequence_length + num_tokens, self.block_size) - len(st.block_table)
        if self._needs_copy(st):
            need += 1
        if need > len(self.free_blocks):
            raise OracleError("OOM", f"need {need} blocks, {len(self.free_blocks)} free")
        return [self.append_slot_for_decode(seq_id) for _ in range(num_tokens)]

    # -- release ---------------------------------------------------------------
    def free_sequence(self, seq_id: int) -> None:
        if seq_id not in self.sequences:
            if seq_id in self.released_ids:
                raise OracleError("DOUBLE_FREE", f"sequence {seq_id} already released")
            raise OracleError("UNKNOWN_SEQ", f"sequence {seq_id} is not live")
        table = self.sequences[seq_id].block_table
        if len(set(table)) != len(table):
            raise OracleError("INVARIANT", "duplicate block in table")
        if any(b < 0 or b >= self.num_blocks for b in table):
            raise OracleError("INVARIANT", "block index out of range")
        if any(self.ref_count[b] == 0 for b in table):
            raise OracleError("INVARIANT", "table holds a free block")
        for b in table:
            self.ref_count[b] -= 1
            if self.ref_count[b] == 0:
                self.free_blocks.append(b)
        del self.sequences[seq_id]
        self.released_ids.add(seq_id)

    # -- invariants --------------------------------------------------------------
    def invariants_ok(self) -> bool:
        bs = self.block_size
        refs: Dict[int, int] = {}
        for st in self.sequences.values():
            if len(st.block_table) != _ceil_div(st.sequence_length, bs):
                return False
            if len(set(st.block_table)) != len(st.block_table):
                return False
            for b in st.block_table:
                if b < 0 or b >= self.num_blocks:
                    return False
                refs[b] = refs.get(b, 0) + 1
        for b in range(self.num_blocks):
            if self.ref_count[b] != refs.get(b, 0):
                return False
        free = self.free_blocks
        if len(set(free)) != len(free) or any(refs.get(b, 0) for b in free):
            return False
        return len(refs) + len(free) == self.num_blocks
