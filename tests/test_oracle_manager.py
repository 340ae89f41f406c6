"""Pins for the oracle block manager: the values the pages print, plus
invariants after every operation of seeded random op sequences."""

import random

import pytest

from oracle.block_manager import BlockManager, OracleError
from oracle.ledger import allocation_report, kv_cache_bytes, tail_waste
from oracle.paged_cache import (block_offset, logical_block, num_logical_blocks, slot_of,
                                split_slot)
from tests.conftest import load_golden

G_MAP = load_golden("address_mapping.json")
G_VLLM = load_golden("mini_vllm_block_manager.json")
G_CH22 = load_golden("llm_algo_ch22.json")


# -- MiniPaged-Qwen worked examples ------------------------------------------------

def test_mapping_worked_example():
    g = G_MAP["mapping_example"]
    bs, pos = g["block_size"], g["token_pos"]
    assert logical_block(pos, bs) == g["logical_block"]
    assert block_offset(pos, bs) == g["block_offset"]
    assert g["table"][logical_block(pos, bs)] == g["physical_block"]
    assert slot_of(g["table"], pos, bs) == g["slot"]


def test_mapping_rows():
    g = G_MAP["mapping_rows"]
    for pos, lb, off in zip(g["token_pos"], g["logical_block"], g["block_offset"]):
        assert (logical_block(pos, g["block_size"]), block_offset(pos, g["block_size"])) == (lb, off)


def test_append_boundary_and_new_block():
    g = G_MAP["append_boundary"]
    bs = g["block_size"]
    for c in g["cases"]:
        # a sequence of length L holds ceil(L / bs) blocks; the next write
        # needs a new one exactly when its logical block equals that count
        m = BlockManager(16, bs)
        m.allocate_for_prefill(0, c["sequence_length"])
        before = len(m.block_table(0))
        slot = m.append_slot_for_decode(0)
        assert (len(m.block_table(0)) > before) == c["needs_new_block"]
        table = m.block_table(0)
        assert slot == table[c["logical_block"]] * bs + c["block_offset"]
    g = G_MAP["append_new_block"]
    bs = g["block_size"]
    # table [5, 2] of a length-8 sequence; the free list offers block 9 first
    order = [5, 2, 9] + [b for b in range(16) if b not in (5, 2, 9)]
    m = BlockManager(16, bs, order)
    m.allocate_for_prefill(7, 8)
    assert m.block_table(7) == g["table_before"]
    slot = m.append_slot_for_decode(7)
    assert m.block_table(7) == g["table_after"]
    assert slot == g["slot"]
    assert split_slot(slot, bs) == (g["physical_block"], g["block_offset"])


def test_slot_decomposition():
    g = G_MAP["slot_decomposition"]
    for c in g["cases"]:
        assert split_slot(c["slot"], g["block_size"]) == (c["physical_block"], c["block_offset"])


def test_block_counts_and_waste():
    g = G_MAP["num_logical_blocks"]
    assert num_logical_blocks(g["sequence_length"], g["block_size"]) == g["blocks"]
    for c in G_MAP["tail_waste"]["cases"]:
        assert num_logical_blocks(c["sequence_length"], c["block_size"]) == c["blocks"]
        assert tail_waste(c["sequence_length"], c["block_size"]) == c["waste"]
    g = G_MAP["max_length_utilisation"]
    r = allocation_report(g["seq_len"], 1, g["reserved"])
    assert round(r["utilization"], 3) == g["utilisation_rounded_3"]


# -- mini-vLLM Block Manager examples ------------------------------------------------

def test_prefill_example():
    g = G_VLLM["prefill_example"]
    n = 16
    order = g["free_before"] + [b for b in range(n) if b not in g["free_before"]]
    m = BlockManager(n, g["block_size"], order)
    m.allocate_for_prefill(0, g["prompt_len"])
    assert m.block_table(0) == g["table"]
    assert m.free_blocks[:len(g["free_after"])] == g["free_after"]


def test_prompt_slots_and_decode_append():
    g = G_VLLM["prompt_slots"]
    bs = g["block_size"]
    order = [3, 8, 1, 5, 7] + [b for b in range(16) if b not in (3, 8, 1, 5, 7)]
    m = BlockManager(16, bs, order)
    slots = m.allocate_for_prefill(0, 40)
    table = m.block_table(0)
    for c in g["cases"]:
        assert slots[c["token"]] == table[c["logical_block"]] * bs + c["block_offset"]
    g = G_VLLM["decode_append"]
    for c in g["cases"]:
        while m.seq_len(0) < c["token"]:
            m.append_slot_for_decode(0)
        before = len(m.block_table(0))
        slot = m.append_slot_for_decode(0)
        assert (len(m.block_table(0)) > before) == c["needs_new_block"]
        assert slot == m.block_table(0)[c["logical_block"]] * bs + c["block_offset"]
    # the block taken at token 48 is the next one on the free list: 5
    assert m.block_table(0) == [3, 8, 1, 5]


def test_scheduler_block_counts():
    g = G_VLLM["scheduler_blocks"]
    m = BlockManager(7, g["block_size"])
    assert m.can_allocate(g["prompt_len"])
    m.allocate_for_prefill(0, g["prompt_len"])
    assert len(m.block_table(0)) == g["blocks"]
    assert not BlockManager(6, g["block_size"]).can_allocate(g["prompt_len"])
    bs = g["block_size"]
    for L in g["boundary_lengths"]:
        m = BlockManager(8, bs)
        m.allocate_for_prefill(0, L)
        before = len(m.block_table(0))
        m.append_slot_for_decode(0)
        assert len(m.block_table(0)) == before + 1
        m2 = BlockManager(8, bs)
        m2.allocate_for_prefill(0, L - 1)
        before = len(m2.block_table(0))
        m2.append_slot_for_decode(0)
        assert len(m2.block_table(0)) == before


def test_lifecycle_example():
    g = G_VLLM["lifecycle"]
    bs = g["block_size"]
    order = g["free_order_prefix"] + [b for b in range(12) if b not in g["free_order_prefix"]]
    m = BlockManager(12, bs, order)
    slots = m.allocate_for_prefill(1, g["prompt_len"])
    assert m.block_table(1) == g["prefill_table"]
    assert [list(split_slot(s, bs)) for s in slots] == g["prompt_rows"]
    rows = [list(split_slot(m.append_slot_for_decode(1), bs)) for _ in g["decode_rows"]]
    assert rows == g["decode_rows"]
    assert m.block_table(1) == g["final_table"]
    assert m.seq_len(1) == g["prompt_len"] + len(g["decode_rows"])


# -- LLM-algo ch.22 tests ------------------------------------------------------------

def test_request_validation():
    for sid, n in G_CH22["request_validation"]["rejected"]:
        with pytest.raises(OracleError) as e:
            BlockManager(4, 4).allocate_for_prefill(sid, n)
        assert e.value.code == "INVALID_ARG"


def test_prefill_decode_case1():
    g = G_CH22["prefill_decode"]
    m = BlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(1, g["prompt_len"])
    assert len(m.block_table(1)) == g["after_prefill"]["blocks"]
    assert m.num_free_blocks() == g["after_prefill"]["free"]
    with pytest.raises(OracleError) as e:
        m.allocate_for_prefill(1, g["prompt_len"])
    assert e.value.code == "DUPLICATE_SEQ"
    m.append_slot_for_decode(1)
    assert len(m.block_table(1)) == g["after_decode_1"]["blocks"]
    m.append_slot_for_decode(1)
    m.append_slot_for_decode(1)
    assert len(m.block_table(1)) == g["after_decode_3"]["blocks"]
    assert m.num_free_blocks() == g["after_decode_3"]["free"]
    assert m.seq_len(1) == g["after_decode_3"]["seq_len"]


def test_oom_and_atomic_oom():
    g = G_CH22["oom"]
    with pytest.raises(OracleError) as e:
        BlockManager(g["num_blocks"], g["block_size"]).allocate_for_prefill(3, g["prompt_len"])
    assert e.value.code == "OOM"
    g = G_CH22["atomic_oom"]
    m = BlockManager(g["num_blocks"], g["block_size"])
    before = list(m.free_blocks)
    with pytest.raises(OracleError) as e:
        m.allocate_for_prefill(4, g["prompt_len"])
    assert e.value.code == "OOM"
    assert m.free_blocks == before and 4 not in m.sequences


def test_ledger():
    g = G_CH22["ledger"]
    r = kv_cache_bytes(g["num_blocks"], g["block_size"], g["num_layers"], g["num_kv_heads"],
                       g["head_dim"], g["dtype_bytes"])
    assert r["kv_bytes_per_token"] == g["kv_bytes_per_token"]
    assert r["total_cache_bytes"] == g["total_cache_bytes"]


def test_report_release_reuse():
    g = G_CH22["report_release"]
    m = BlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(5, g["prompt_len"])
    r = allocation_report(m.seq_len(5), len(m.block_table(5)), g["block_size"])
    assert r["allocated_tokens"] == g["allocated_tokens"]
    assert r["unused_tail_tokens"] == g["unused_tail_tokens"]
    assert round(r["utilization"], 3) == g["utilization"]
    m.free_sequence(5)
    assert 5 not in m.sequences
    # the page sorts on release; our policy does not, so compare as sets
    assert sorted(m.free_blocks) == g["free_after_release"]
    with pytest.raises(OracleError) as e:
        m.free_sequence(5)
    assert e.value.code == "DOUBLE_FREE"
    # released blocks are reusable
    m.allocate_for_prefill(6, g["num_blocks"] * g["block_size"])
    assert sorted(m.block_table(6)) == [0, 1, 2]


def test_decode_rollback():
    g = G_CH22["decode_rollback"]
    m = BlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(6, g["prompt_len"])
    table = m.block_table(6)
    with pytest.raises(OracleError) as e:
        m.append_slot_for_decode(6)
    assert e.value.code == "OOM"
    assert m.seq_len(6) == g["seq_len_after"] and m.block_table(6) == table


# -- extra semantics ----------------------------------------------------------------

def test_errors_and_batched_ops():
    m = BlockManager(4, 4)
    with pytest.raises(OracleError) as e:
        m.append_slot_for_decode(9)
    assert e.value.code == "UNKNOWN_SEQ"
    with pytest.raises(OracleError) as e:
        m.free_sequence(9)
    assert e.value.code == "UNKNOWN_SEQ"
    m.allocate_for_prefill(0, 3)
    m.allocate_for_prefill(1, 4)
    # decode step: seq 0 stays in its block, seq 1 needs one more
    free_before = list(m.free_blocks)
    slots = m.decode_step([0, 1])
    assert slots[0] == m.block_table(0)[0] * 4 + 3
    assert slots[1] == m.block_table(1)[1] * 4 + 0
    assert m.free_blocks == free_before[1:]
    # append_slots across a boundary is all-or-nothing
    m2 = BlockManager(2, 4)
    m2.allocate_for_prefill(0, 2)
    with pytest.raises(OracleError):
        m2.append_slots(0, 7)          # needs 3 blocks in total, pool has 2
    assert m2.seq_len(0) == 2 and len(m2.block_table(0)) == 1
    assert m2.append_slots(0, 6) == [m2.block_table(0)[p // 4] * 4 + p % 4 for p in range(2, 8)]
    with pytest.raises(OracleError) as e:
        m.decode_step([0, 0])
    assert e.value.code == "INVALID_ARG"


def test_decode_step_atomic_oom():
    m = BlockManager(3, 2)
    m.allocate_for_prefill(0, 2)     # full block: next append needs a block
    m.allocate_for_prefill(1, 2)
    m.allocate_for_prefill(2, 1)     # fills the pool
    st = {s: (m.seq_len(s), m.block_table(s)) for s in (0, 1, 2)}
    with pytest.raises(OracleError) as e:
        m.decode_step([2, 0])
    assert e.value.code == "OOM"
    assert {s: (m.seq_len(s), m.block_table(s)) for s in (0, 1, 2)} == st


def test_invariants_detect_corruption():
    m = BlockManager(8, 2)
    m.allocate_for_prefill(0, 3)
    m.allocate_for_prefill(1, 3)
    assert m.invariants_ok()
    m.sequences[1].block_table[0] = m.sequences[0].block_table[0]   # two owners
    assert not m.invariants_ok()
    m = BlockManager(8, 2)
    m.allocate_for_prefill(0, 3)
    m.free_blocks.append(m.sequences[0].block_table[1])             # allocated and free
    assert not m.invariants_ok()
    with pytest.raises(OracleError) as e:
        m.free_sequence(0)
    assert e.value.code == "INVARIANT"
    m = BlockManager(8, 2)
    m.allocate_for_prefill(0, 3)
    m.sequences[0].sequence_length = 5                              # length beyond the tail
    assert not m.invariants_ok()
    m = BlockManager(8, 2)
    m.allocate_for_prefill(0, 3)
    m.free_blocks.pop()                                             # a lost block
    assert not m.invariants_ok()


def _owner_table(m):
    owner = [None] * m.num_blocks
    for sid, st in m.sequences.items():
        for b in st.block_table:
            assert owner[b] is None
            owner[b] = sid
    for b in m.free_blocks:
        assert owner[b] is None
    return owner


@pytest.mark.parametrize("seed", range(6))
def test_random_ops_keep_invariants(seed):
    """mini-vLLM "正确性不变量": after every operation the owner table is
    consistent, tables follow logical order, lengths match tails."""
    rng = random.Random(seed)
    nb, bs = rng.choice([(8, 1), (16, 2), (32, 4), (64, 16)])
    order = list(range(nb))
    rng.shuffle(order)
    m = BlockManager(nb, bs, order)
    next_id = 0
    logical = {}   # seq -> list of (slot) by position, to check table order
    for _ in range(400):
        op = rng.random()
        live = list(m.sequences)
        try:
            if op < 0.3 or not live:
                n = rng.randint(1, 3 * bs)
                slots = m.allocate_for_prefill(next_id, n)
                logical[next_id] = slots
                next_id += 1
            elif op < 0.75:
                sid = rng.choice(live)
                logical[sid].append(m.append_slot_for_decode(sid))
            elif op < 0.85:
                sid = rng.choice(live)
                logical[sid].extend(m.append_slots(sid, rng.randint(1, 2 * bs)))
            else:
                sid = rng.choice(live)
                m.free_sequence(sid)
                del logical[sid]
        except OracleError as e:
            assert e.code == "OOM"
        assert m.invariants_ok()
        _owner_table(m)
        for sid, slots in logical.items():
            table = m.block_table(sid)
            assert len(slots) == m.seq_len(sid)
            assert slots == [slot_of(table, p, bs) for p in range(len(slots))]
