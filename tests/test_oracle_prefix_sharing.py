"""Pins for the sharing oracle (prefix sharing and copy-on-write,
"paged-attention-impl-detail", section Copy-on-Write共享), and the native
manager against it.

What pins the oracle, independently of its own code:
* the page's two rules, stated on small cases: a shared block counts its
  holders (share_prefix_blocks); a writer to a block held by others takes a
  fresh block, the old count drops by one and the new block's count is 1,
  while a sole holder writes in place (copy_on_write);
* a content simulation: every append writes a unique tag at its slot in a
  simulated pool, queued copies move whole blocks first, and every live
  sequence, read back through its table, must give exactly its own tokens
  (the parent's first prefix_len tokens, then its own appends);
* with no fork, the sharing manager behaves exactly as the pinned base
  manager (same slots, tables, free lists, errors).
"""

import random

import numpy as np
import pytest

from oracle.block_manager import BlockManager, OracleError
from oracle.prefix_sharing import SharingBlockManager
from paged_kv_cache_128_gb300 import KVBlockManager, KVError


def test_fork_counts_holders_and_takes_no_block():
    m = SharingBlockManager(8, 4)
    m.allocate_for_prefill(0, 10)            # 3 blocks: [0, 1, 2]
    assert m.block_table(0) == [0, 1, 2]
    m.fork(0, 1, 10)
    m.fork(0, 2, 5)                          # ceil(5 / 4) = 2 shared blocks
    assert m.block_table(1) == [0, 1, 2] and m.seq_len(1) == 10
    assert m.block_table(2) == [0, 1] and m.seq_len(2) == 5
    assert m.ref_count[:4] == [3, 3, 2, 0]
    assert m.num_free_blocks() == 5
    assert m.invariants_ok()


def test_copy_on_write_rule():
    m = SharingBlockManager(8, 4)
    m.allocate_for_prefill(0, 10)            # [0, 1, 2], block 2 holds positions 8, 9
    m.fork(0, 1, 10)
    slot = m.append_slot_for_decode(1)       # position 10 lands in shared block 2
    assert m.take_copies() == [(2, 3)]       # fresh block from the front of the free list
    assert m.block_table(1) == [0, 1, 3] and slot == 3 * 4 + 2
    assert m.ref_count[2] == 1 and m.ref_count[3] == 1
    slot = m.append_slot_for_decode(0)       # now the sole holder of block 2: in place
    assert m.take_copies() == [] and slot == 2 * 4 + 2
    assert m.block_table(0) == [0, 1, 2]
    assert m.invariants_ok()


def test_fork_at_block_boundary_needs_no_copy():
    m = SharingBlockManager(8, 4)
    m.allocate_for_prefill(0, 8)
    m.fork(0, 1, 8)
    m.append_slot_for_decode(1)              # position 8 opens a new block
    m.append_slot_for_decode(0)
    assert m.take_copies() == []
    assert m.block_table(0)[:2] == m.block_table(1)[:2] and m.block_table(0)[2] != m.block_table(1)[2]


def test_release_frees_a_shared_block_with_its_last_holder():
    m = SharingBlockManager(6, 4)
    m.allocate_for_prefill(0, 6)             # [0, 1]
    m.fork(0, 1, 6)
    m.free_sequence(0)
    assert m.num_free_blocks() == 4 and m.ref_count[:2] == [1, 1]
    m.free_sequence(1)
    assert m.free_blocks == [2, 3, 4, 5, 0, 1]
    with pytest.raises(OracleError) as e:
        m.free_sequence(1)
    assert e.value.code == "DOUBLE_FREE"


def test_copy_needs_a_free_block_and_fails_atomically():
    m = SharingBlockManager(2, 4)
    m.allocate_for_prefill(0, 3)
    m.fork(0, 1, 3)
    m.allocate_for_prefill(2, 4)             # pool now full
    assert not m.can_append_slots([1])
    with pytest.raises(OracleError) as e:
        m.append_slot_for_decode(1)
    assert e.value.code == "OOM"
    assert m.block_table(1) == [0] and m.seq_len(1) == 3 and m.take_copies() == []
    with pytest.raises(OracleError):
        m.append_slots(0, 2)
    assert m.invariants_ok()


def test_fork_validation():
    m = SharingBlockManager(4, 4)
    m.allocate_for_prefill(0, 5)
    for args, code in (((9, 1, 2), "UNKNOWN_SEQ"), ((0, 0, 2), "DUPLICATE_SEQ"), ((0, 1, 0), "INVALID_ARG"),
                       ((0, 1, 6), "INVALID_ARG"), ((0, -1, 2), "INVALID_ARG")):
        with pytest.raises(OracleError) as e:
            m.fork(*args)
        assert e.value.code == code


def test_planted_refcount_error_is_caught():
    m = SharingBlockManager(8, 4)
    m.allocate_for_prefill(0, 6)
    m.fork(0, 1, 6)
    assert m.invariants_ok()
    m.ref_count[0] -= 1
    assert not m.invariants_ok()


def _simulate(mgr, rng, n_ops, tags=True):
    """Random prefills, forks, appends and releases; every live sequence must
    read back its own tokens through its table from the simulated pool."""
    bs = mgr.block_size
    pool = {}                                # slot -> tag
    logical = {}                             # seq -> list of tags
    next_id = 0

    def apply_copies():
        for src, dst in mgr.take_copies():
            for off in range(bs):
                if src * bs + off in pool:
                    pool[dst * bs + off] = pool[src * bs + off]
                else:
                    pool.pop(dst * bs + off, None)

    for step in range(n_ops):
        live = list(mgr.sequences)
        r = rng.random()
        try:
            if r < 0.2 or not live:
                n = rng.randint(1, 3 * bs)
                slots = mgr.allocate_for_prefill(next_id, n)
                logical[next_id] = [(next_id, t) for t in range(n)]
                for t, s in enumerate(slots):
                    pool[s] = logical[next_id][t]
                next_id += 1
            elif r < 0.4:
                parent = rng.choice(live)
                plen = rng.randint(1, mgr.seq_len(parent))
                mgr.fork(parent, next_id, plen)
                logical[next_id] = logical[parent][:plen]
                next_id += 1
            elif r < 0.85:
                sid = rng.choice(live)
                k = rng.randint(1, 3)
                slots = mgr.append_slots(sid, k)
                apply_copies()                 # copies precede the writes
                for s in slots:
                    tag = (sid, len(logical[sid]), step)
                    logical[sid].append(tag)
                    pool[s] = tag
            else:
                sid = rng.choice(live)
                mgr.free_sequence(sid)
                del logical[sid]
        except OracleError as e:
            assert e.code == "OOM"
            assert mgr.take_copies() == []
        assert mgr.invariants_ok()
        for sid, st in mgr.sequences.items():
            got = [pool.get(st.block_table[p // bs] * bs + p % bs) for p in range(st.sequence_length)]
            assert got == logical[sid], f"sequence {sid} reads back wrong tokens"


@pytest.mark.parametrize("seed", range(6))
def test_content_simulation(seed):
    rng = random.Random(seed)
    order = list(range(24))
    rng.shuffle(order)
    _simulate(SharingBlockManager(24, rng.choice([1, 2, 4, 8]), order), rng, 400)


@pytest.mark.parametrize("seed", range(4))
def test_without_forks_equals_base_manager(seed):
    rng = random.Random(100 + seed)
    order = list(range(32))
    rng.shuffle(order)
    a, b = BlockManager(32, 4, order), SharingBlockManager(32, 4, order)
    live, nid = [], 0
    for _ in range(300):
        r = rng.random()
        op = ("prefill", nid, rng.randint(1, 20)) if r < 0.3 or not live else \
            ("append", rng.choice(live), rng.randint(1, 5)) if r < 0.8 else ("free", rng.choice(live), 0)
        res = []
        for m in (a, b):
            try:
                if op[0] == "prefill":
                    res.append(m.allocate_for_prefill(op[1], op[2]))
                elif op[0] == "append":
                    res.append(m.append_slots(op[1], op[2]))
                else:
                    res.append(m.free_sequence(op[1]))
            except OracleError as e:
                res.append(e.code)
        assert res[0] == res[1]
        if op[0] == "prefill" and not isinstance(res[0], str):
            live.append(nid)
            nid += 1
        if op[0] == "free":
            live.remove(op[1])
        assert a.free_blocks == b.free_blocks
        assert {s: t.block_table for s, t in a.sequences.items()} == {s: t.block_table for s, t in b.sequences.items()}
    assert b.take_copies() == []


# ---------------------------------------------------------------- native manager

def _native_op(nat, op):
    kind = op[0]
    if kind == "prefill":
        return nat.allocate_for_prefill(op[1], op[2]).tolist()
    if kind == "fork":
        return nat.fork(op[1], op[2], op[3])
    if kind == "append":
        return nat.append_slots(op[1], op[2]).tolist()
    if kind == "decode":
        return nat.decode_step(op[1], op[2])[0].tolist()
    return nat.free_sequence(op[1])


def _oracle_op(ora, op):
    kind = op[0]
    if kind == "prefill":
        return ora.allocate_for_prefill(op[1], op[2])
    if kind == "fork":
        return ora.fork(op[1], op[2], op[3])
    if kind == "append":
        return ora.append_slots(op[1], op[2])
    if kind == "decode":
        return ora.decode_step(op[1])
    return ora.free_sequence(op[1])


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_sharing_oracle(seed):
    rng = random.Random(7000 + seed)
    nb, bs = 40, rng.choice([2, 4, 16])
    order = list(range(nb))
    rng.shuffle(order)
    nat, ora = KVBlockManager(nb, bs, order), SharingBlockManager(nb, bs, order)
    nid = 0
    for _ in range(400):
        live = sorted(ora.sequences)
        r = rng.random()
        if r < 0.15 or not live:
            op = ("prefill", nid, rng.randint(1, 4 * bs))
        elif r < 0.35:
            p = rng.choice(live)
            op = ("fork", p, nid, rng.randint(1, ora.seq_len(p)))
        elif r < 0.6:
            op = ("append", rng.choice(live), rng.randint(1, 3))
        elif r < 0.85:
            op = ("decode", rng.sample(live, rng.randint(1, len(live))), 4 * bs + 64)
        else:
            op = ("free", rng.choice(live))
        try:
            want, err_o = _oracle_op(ora, op), None
        except OracleError as e:
            want, err_o = None, e.code
        try:
            got, err_n = _native_op(nat, op), None
        except KVError as e:
            got, err_n = None, e.code
        assert err_n == err_o, op
        if err_o is None:
            assert got == want, op
            if op[0] in ("prefill", "fork"):
                nid += 1
        src, dst = nat.take_copies()
        assert list(zip(src.tolist(), dst.tolist())) == ora.take_copies()
        assert nat.free_list().tolist() == ora.free_blocks
        for sid, st in ora.sequences.items():
            assert nat.block_table(sid).tolist() == st.block_table
            assert nat.seq_len(sid) == st.sequence_length
        assert [nat.block_refcount(b) for b in range(nb)] == ora.ref_count
        assert nat.check_invariants() and ora.invariants_ok()
        owner = nat.owner_table()
        for b in range(nb):
            holders = [s for s, st in ora.sequences.items() if b in st.block_table]
            assert owner[b] == (-1 if not holders else holders[0] if len(holders) == 1 else -2)


def test_native_fork_codes_and_copy_queue():
    nat = KVBlockManager(8, 4)
    nat.allocate_for_prefill(0, 10)
    for args, code in (((9, 1, 2), "UNKNOWN_SEQ"), ((0, 0, 2), "DUPLICATE_SEQ"), ((0, 1, 0), "INVALID_ARG"),
                       ((0, 1, 11), "INVALID_ARG")):
        with pytest.raises(KVError) as e:
            nat.fork(*args)
        assert e.value.code == code
    nat.fork(0, 1, 10)
    nat.append_slot_for_decode(1)
    nat.append_slot_for_decode(0)
    src, dst = nat.take_copies()
    assert src.tolist() == [2] and dst.tolist() == [3]
    assert nat.take_copies()[0].size == 0
