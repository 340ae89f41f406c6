"""The native (C++) block manager against the oracle manager, on CPU.

Block tables, free lists, slots and error codes must be bit-exact: the same
seeded operations go to both, and every result and the full state are
compared after each one.  Also: the pages' worked examples run directly on
the native manager, and every workload's setup replays identically."""

import random

import numpy as np
import pytest

from oracle.block_manager import BlockManager as OracleManager
from oracle.block_manager import OracleError
from oracle.ledger import kv_cache_bytes
from paged_kv_cache_128_gb300 import KVBlockManager, KVError, kv_cache_ledger
from paged_kv_cache_128_gb300.inputs import WORKLOADS, make_workload
from tests.conftest import load_golden

G_CH22 = load_golden("llm_algo_ch22.json")
G_VLLM = load_golden("mini_vllm_block_manager.json")
G_MAP = load_golden("address_mapping.json")


def _same_state(nat: KVBlockManager, ora: OracleManager):
    assert nat.free_list().tolist() == ora.free_blocks
    assert nat.num_free_blocks() == len(ora.free_blocks)
    for sid, st in ora.sequences.items():
        assert nat.block_table(sid).tolist() == st.block_table
        assert nat.seq_len(sid) == st.sequence_length
    assert nat.stats()["num_sequences"] == len(ora.sequences)
    assert nat.check_invariants() and ora.invariants_ok()
    owner = nat.owner_table()
    want = np.full(ora.num_blocks, -1, dtype=np.int64)
    for sid, st in ora.sequences.items():
        want[st.block_table] = sid
    assert np.array_equal(owner, want)


def _both(fn_nat, fn_ora):
    """Run one op on both; results equal, or both fail with the same code."""
    try:
        r_o = fn_ora()
        err_o = None
    except OracleError as e:
        err_o = e.code
    try:
        r_n = fn_nat()
        err_n = None
    except KVError as e:
        err_n = e.code
    assert err_n == err_o
    if err_o is None:
        if isinstance(r_n, np.ndarray):
            r_n = r_n.tolist()
        assert r_n == r_o


@pytest.mark.parametrize("seed", range(8))
def test_random_ops_match_oracle(seed):
    rng = random.Random(100 + seed)
    nb, bs = rng.choice([(8, 1), (16, 2), (24, 4), (64, 16), (33, 5)])
    order = list(range(nb))
    rng.shuffle(order)
    nat, ora = KVBlockManager(nb, bs, order), OracleManager(nb, bs, order)
    next_id = 0
    for _ in range(300):
        live = list(ora.sequences)
        r = rng.random()
        if r < 0.25 or not live:
            n = rng.randint(-1, 3 * bs)
            sid = next_id if rng.random() < 0.9 else rng.choice(live + [next_id])
            _both(lambda: nat.allocate_for_prefill(sid, n), lambda: ora.allocate_for_prefill(sid, n))
            if sid in ora.sequences and sid == next_id:
                next_id += 1
        elif r < 0.55:
            sid = rng.choice(live + [10_000])
            _both(lambda: nat.append_slot_for_decode(sid), lambda: ora.append_slot_for_decode(sid))
        elif r < 0.65:
            sid = rng.choice(live)
            n = rng.randint(0, 2 * bs)
            _both(lambda: nat.append_slots(sid, n), lambda: ora.append_slots(sid, n))
        elif r < 0.8:
            ids = rng.sample(live, rng.randint(1, len(live)))
            if rng.random() < 0.1:
                ids = ids + ids[:1]
            mb = max(len(ora.sequences[s].block_table) for s in ids) + 2 if all(s in ora.sequences for s in ids) else 4

            def nat_step():
                slots, tables, lens = nat.decode_step(ids, mb)
                return [slots.tolist(), tables.tolist(), lens.tolist()]

            def ora_step():
                slots = ora.decode_step(ids)
                tables, lens = ora.export(ids, mb)
                return [slots, tables, lens]

            _both(nat_step, ora_step)
        elif r < 0.9:
            sid = rng.choice(live + [next_id + 50])
            _both(lambda: nat.free_sequence(sid), lambda: ora.free_sequence(sid))
        else:
            ids = rng.sample(live, rng.randint(1, len(live)))
            _both(lambda: nat.can_append_slots(ids), lambda: ora.can_append_slots(ids))
            n = rng.randint(1, 5 * bs)
            _both(lambda: nat.can_allocate(n), lambda: ora.can_allocate(n))
        _same_state(nat, ora)


def test_double_free_and_reuse_codes():
    nat = KVBlockManager(3, 4)
    nat.allocate_for_prefill(5, 5)
    nat.free_sequence(5)
    with pytest.raises(KVError) as e:
        nat.free_sequence(5)
    assert e.value.code == "DOUBLE_FREE"
    with pytest.raises(KVError) as e:
        nat.free_sequence(6)
    assert e.value.code == "UNKNOWN_SEQ"
    nat.allocate_for_prefill(5, 12)            # a released id may be prefilled again
    assert sorted(nat.block_table(5).tolist()) == [0, 1, 2]


@pytest.mark.parametrize("seed", range(4))
def test_release_and_reprefill_codes_match_oracle(seed):
    """Ids from a small universe are prefilled, released, released again
    and prefilled again in random order, so the released-id ranges merge
    and split often; every result and error code must equal the oracle's
    (which remembers released ids in a plain set)."""
    rng = random.Random(700 + seed)
    nat, ora = KVBlockManager(256, 1), OracleManager(256, 1)
    for _ in range(1500):
        sid = rng.randrange(40)
        if rng.random() < 0.5:
            _both(lambda: nat.allocate_for_prefill(sid, 1), lambda: ora.allocate_for_prefill(sid, 1))
        else:
            _both(lambda: nat.free_sequence(sid), lambda: ora.free_sequence(sid))
        _same_state(nat, ora)


def test_released_ids_are_kept_as_ranges():
    nat = KVBlockManager(512, 1)
    for sid in range(300):
        nat.allocate_for_prefill(sid, 1)
    for sid in range(300):                    # released in order: one range
        nat.free_sequence(sid)
    assert nat.released_ranges() == 1
    for sid in (0, 150, 299):
        with pytest.raises(KVError) as e:
            nat.free_sequence(sid)
        assert e.value.code == "DOUBLE_FREE"
    with pytest.raises(KVError) as e:
        nat.free_sequence(300)
    assert e.value.code == "UNKNOWN_SEQ"
    nat.allocate_for_prefill(150, 1)          # prefilled again: the range splits
    assert nat.released_ranges() == 2
    nat.free_sequence(150)
    assert nat.released_ranges() == 1
    for sid in range(400, 500, 2):            # every other id: one range each
        nat.allocate_for_prefill(sid, 1)
        nat.free_sequence(sid)
    assert nat.released_ranges() == 51
    for sid in range(401, 500, 2):            # the gaps filled: merged into one
        nat.allocate_for_prefill(sid, 1)
        nat.free_sequence(sid)
    assert nat.released_ranges() == 2


def test_pages_examples_on_native():
    g = G_CH22["prefill_decode"]
    m = KVBlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(1, g["prompt_len"])
    assert m.num_free_blocks() == g["after_prefill"]["free"]
    with pytest.raises(KVError) as e:
        m.allocate_for_prefill(1, g["prompt_len"])
    assert e.value.code == "DUPLICATE_SEQ"
    for _ in range(3):
        m.append_slot_for_decode(1)
    assert len(m.block_table(1)) == g["after_decode_3"]["blocks"] and m.num_free_blocks() == 7
    for sid, n in G_CH22["request_validation"]["rejected"]:
        with pytest.raises(KVError) as e:
            KVBlockManager(4, 4).allocate_for_prefill(sid, n)
        assert e.value.code == "INVALID_ARG"
    g = G_CH22["atomic_oom"]
    m = KVBlockManager(g["num_blocks"], g["block_size"])
    before = m.free_list().tolist()
    with pytest.raises(KVError) as e:
        m.allocate_for_prefill(4, g["prompt_len"])
    assert e.value.code == "OOM" and m.free_list().tolist() == before
    g = G_CH22["decode_rollback"]
    m = KVBlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(6, g["prompt_len"])
    with pytest.raises(KVError) as e:
        m.append_slot_for_decode(6)
    assert e.value.code == "OOM" and m.seq_len(6) == g["seq_len_after"]
    g = G_CH22["report_release"]
    m = KVBlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(5, g["prompt_len"])
    r = m.allocation_report(5)
    assert (r["allocated_tokens"], r["unused_tail_tokens"], round(r["utilization"], 3)) == (8, 3, 0.625)
    g = G_VLLM["lifecycle"]
    order = g["free_order_prefix"] + [b for b in range(12) if b not in g["free_order_prefix"]]
    m = KVBlockManager(12, g["block_size"], order)
    slots = m.allocate_for_prefill(1, g["prompt_len"])
    assert [[s // 4, s % 4] for s in slots] == g["prompt_rows"]
    got = [m.append_slot_for_decode(1) for _ in g["decode_rows"]]
    assert [[s // 4, s % 4] for s in got] == g["decode_rows"]
    g = G_MAP["append_new_block"]
    order = [5, 2, 9] + [b for b in range(16) if b not in (5, 2, 9)]
    m = KVBlockManager(16, 4, order)
    m.allocate_for_prefill(0, 8)
    assert m.append_slot_for_decode(0) == g["slot"]


def test_ledger_native_matches_pages_and_oracle():
    g = G_CH22["ledger"]
    args = (g["num_blocks"], g["block_size"], g["num_layers"], g["num_kv_heads"], g["head_dim"], g["dtype_bytes"])
    r = kv_cache_ledger(*args)
    assert r["kv_bytes_per_token"] == g["kv_bytes_per_token"] and r["total_cache_bytes"] == g["total_cache_bytes"]
    assert r == kv_cache_bytes(*args)


def test_create_rejects_bad_free_order():
    for order in ([0, 1, 1, 3], [0, 1, 2, 4], [0, 1, 2]):
        with pytest.raises(KVError) as e:
            KVBlockManager(4, 2, order)
        assert e.value.code == "INVALID_ARG"
    with pytest.raises(KVError):
        KVBlockManager(0, 4)
    with pytest.raises(KVError):
        KVBlockManager(1 << 30, 4)      # slots would overflow int32


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_setup_replays_identically(name):
    wl = make_workload(name)
    nat = KVBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
    ora = OracleManager(wl.num_blocks, wl.block_size, None if wl.free_order is None else wl.free_order.tolist())
    for op, sid, n in wl.setup_ops:
        if op == "prefill":
            a, b = nat.allocate_for_prefill(sid, n), ora.allocate_for_prefill(sid, n)
        elif op == "append":
            a, b = nat.append_slots(sid, n), ora.append_slots(sid, n)
        else:
            nat.free_sequence(sid)
            ora.free_sequence(sid)
            continue
        assert a.tolist() == b
    ids = wl.decode_ids.tolist()
    mb = int(wl.cached_lens.max()) // wl.block_size + 4
    slots, tables, lens = nat.decode_step(ids, mb)
    assert slots.tolist() == ora.decode_step(ids)
    t_o, l_o = ora.export(ids, mb)
    assert tables.tolist() == t_o and lens.tolist() == l_o
    assert nat.free_list().tolist() == ora.free_blocks
    assert nat.check_invariants()


def _oracle_prepare(ora, free_ids, pre_ids, pre_lens, dec_ids, pads, mb):
    for s in free_ids:
        ora.free_sequence(s)
    step = []
    for sid, n in zip(pre_ids, pre_lens):
        step += ora.allocate_for_prefill(sid, n)
    step += ora.decode_step(dec_ids)
    total = len(step) + len(pads)
    it = iter(step)
    mapping = [-1 if p in set(pads) else next(it) for p in range(total)]
    tables, lens = ora.export(dec_ids, mb)
    return mapping, tables, lens


@pytest.mark.parametrize("seed", range(6))
def test_prepare_step_matches_oracle_sequence(seed):
    """kvbm_prepare_step = release, prefill each, decode step, pad, export --
    bit-exact against the oracle doing those operations one by one."""
    rng = random.Random(500 + seed)
    nb, bs = rng.choice([(64, 4), (200, 16), (40, 2)])
    order = list(range(nb))
    rng.shuffle(order)
    nat, ora = KVBlockManager(nb, bs, order), OracleManager(nb, bs, order)
    running = []
    for sid in range(6):
        n = rng.randint(1, 3 * bs)
        nat.allocate_for_prefill(sid, n)
        ora.allocate_for_prefill(sid, n)
        running.append(sid)
    next_id, prev = 100, []
    for _ in range(8):
        pre_ids = [next_id + i for i in range(rng.randint(0, 3))]
        next_id += 10
        pre_lens = [rng.randint(1, 2 * bs) for _ in pre_ids]
        n_tot = sum(pre_lens) + len(running)
        n_pad = rng.randint(0, 4)
        pads = sorted(rng.sample(range(n_tot + n_pad), n_pad))
        mb = 64
        try:
            want = _oracle_prepare(ora, prev, pre_ids, pre_lens, running, pads, mb)
            err_o = None
        except OracleError as e:
            err_o = e.code
        try:
            got = nat.prepare_step(prev, pre_ids, pre_lens, running, pads, mb)
            err_n = None
        except KVError as e:
            err_n = e.code
        assert err_n == err_o
        if err_o is None:
            assert got[0].tolist() == want[0]
            assert got[1].tolist() == want[1] and got[2].tolist() == want[2]
            prev = pre_ids
        else:
            break
        _same_state(nat, ora)


def test_prepare_step_is_atomic_and_validates():
    nat = KVBlockManager(4, 4)
    nat.allocate_for_prefill(0, 4)            # full block: the next decode needs one more
    nat.allocate_for_prefill(1, 3)
    before = nat.free_list().tolist()
    with pytest.raises(KVError) as e:          # 2 prefill blocks + 1 decode block > 2 free
        nat.prepare_step([], [7], [8], [0, 1], [], 8)
    assert e.value.code == "OOM"
    assert nat.free_list().tolist() == before and nat.seq_len(0) == 4
    with pytest.raises(KVError) as e:
        nat.prepare_step([], [], [], [0, 1], [0, 0], 8)       # padding positions not increasing
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(KVError) as e:
        nat.prepare_step([], [1], [2], [0], [], 8)            # prefill of a live sequence
    assert e.value.code == "DUPLICATE_SEQ"
    with pytest.raises(KVError) as e:
        nat.prepare_step([], [], [], [0, 0], [], 8)           # one sequence twice
    assert e.value.code == "INVALID_ARG"
    slots, tables, lens = nat.prepare_step([1], [5], [3], [0], [0, 4], 8)
    assert slots.size == 3 + 1 + 2 and slots[0] == -1 and slots[4] == -1
    assert lens.tolist() == [5] and nat.check_invariants()


def test_export_update_equals_full_export():
    """kvbm_export_update keeps a buffer equal to kvbm_export through random
    appends, releases with new sequences in the freed rows, copy-on-write
    forks (the shared last block replaced by the next append) and rows that
    swap sequences, starting from a buffer of garbage."""
    rng = np.random.default_rng(7)
    bs, nb, maxb, R = 4, 1024, 40, 6
    mgr = KVBlockManager(nb, bs)
    next_id = 0
    rows = []
    for _ in range(R):
        mgr.allocate_for_prefill(next_id, int(rng.integers(1, 30)))
        rows.append(next_id)
        next_id += 1
    lens = {sid: mgr.seq_len(sid) for sid in rows}
    tables = np.full((R, maxb), 12345, np.int32)
    prev_ids = np.full(R, -1, np.int64)
    prev_nb = np.zeros(R, np.int32)
    for _ in range(300):
        op = int(rng.integers(0, 5))
        r = int(rng.integers(0, R))
        sid = rows[r]
        if op <= 1 and lens[sid] + 3 <= maxb * bs:              # appends (block growth, copy-on-write)
            n = int(rng.integers(1, 4))
            mgr.append_slots(sid, n)
            lens[sid] += n
        elif op == 2 or lens[sid] + 3 > maxb * bs:               # release, new sequence in the same row
            mgr.free_sequence(sid)
            if sid not in rows[:r] + rows[r + 1:]:
                del lens[sid]
            mgr.allocate_for_prefill(next_id, int(rng.integers(1, 40)))
            rows[r] = next_id
            lens[next_id] = mgr.seq_len(next_id)
            next_id += 1
        elif op == 3:                                              # fork: the child shares the parent's blocks
            child = next_id
            next_id += 1
            mgr.fork(sid, child, lens[sid])
            lens[child] = lens[sid]
            old = rows[(r + 1) % R]
            rows[(r + 1) % R] = child
            if old not in rows:
                mgr.free_sequence(old)
                del lens[old]
        else:                                                      # two rows swap their sequences
            r2 = int(rng.integers(0, R))
            rows[r], rows[r2] = rows[r2], rows[r]
        if len(set(rows)) != R:
            continue
        mgr.export_update(rows, maxb, tables, prev_ids, prev_nb)
        full, _ = mgr.export(rows, maxb)
        assert np.array_equal(tables, full)
    assert mgr.check_invariants()


def test_prepare_step_duplicate_and_unknown_ids():
    """The step's id checks: a new id prefilled twice is DUPLICATE_SEQ; a
    decode id that is one of the step's prefills is INVALID_ARG; a decode id
    never seen is UNKNOWN_SEQ; nothing changes in any of them.  The same
    checks hold call after call (the id set is reused across calls)."""
    nat = KVBlockManager(64, 4)
    nat.allocate_for_prefill(0, 5)
    nat.allocate_for_prefill(1, 2)
    before = (nat.free_list().tolist(), nat.seq_len(0), nat.seq_len(1))
    for _ in range(3):
        for args, code in [(([], [7, 7], [3, 3], [0], [], 8), "DUPLICATE_SEQ"),
                           (([], [7], [3], [0, 7], [], 8), "INVALID_ARG"),
                           (([], [], [], [0, 9], [], 8), "UNKNOWN_SEQ"),
                           (([], [], [], [1, 0, 1], [], 8), "INVALID_ARG")]:
            with pytest.raises(KVError) as e:
                nat.prepare_step(*args)
            assert e.value.code == code, args
            assert (nat.free_list().tolist(), nat.seq_len(0), nat.seq_len(1)) == before
        with pytest.raises(KVError) as e:
            nat.decode_step([1, 1], 8)
        assert e.value.code == "INVALID_ARG"
    slots, tables, lens = nat.prepare_step([], [7], [3], [0, 1], [], 8)
    assert lens.tolist() == [6, 3] and nat.check_invariants()
