"""The opt-in event trace (ag_gemm_plan_set_trace / ag_gemm_plan_trace).

The trace records, per run, when each copy item landed in the staging (just
before its ready counter is released) and when each consumer started and
stopped waiting for remote rows.  Its invariants are the streaming contract of
the method ("AllGather + GEMM 通算融合算子示例", 流式流水线: a chunk is consumed
once it has landed, and the producer sends in consumption order):

* every chunk (fused paths) or chunk k-part (skinny path) lands exactly as
  often as its counter target says;
* a wait ends no earlier than the landing of every chunk (part) it waited for;
* each copy warp lands its items in increasing consumption order;
* a traced run computes exactly what an untraced run does.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from all_gather_gemm_chunked_gb300 import binding as B_  # noqa: E402
from all_gather_gemm_chunked_gb300 import synth  # noqa: E402
from all_gather_gemm_chunked_gb300.plan import Plan  # noqa: E402

DEV = torch.device("cuda:0")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(plan, x, dtype):
    shards = [_dev(s) for s in x["shards"]]
    if dtype == "i8":
        Ci, D = plan.dequant_run(shards, _dev(x["B"]), _dev(x["bias"]), _dev(x["scale"]))
        torch.cuda.synchronize()
        assert plan.status() == 0, f"status word {plan.status_word():#x}"
        return Ci.cpu().numpy(), D.cpu().numpy()
    C = plan.run(shards, _dev(x["B"]))
    torch.cuda.synchronize()
    assert plan.status() == 0, f"status word {plan.status_word():#x}"
    return (C.cpu().numpy(),)


def _check_copy_order(ev):
    landed = ev[ev["kind"] == B_.TRACE_LANDED]
    for key in set(zip(landed["cta"].tolist(), landed["warp"].tolist())):
        mine = landed[(landed["cta"] == key[0]) & (landed["warp"] == key[1])]
        by_item = mine[np.argsort(mine["aux"], kind="stable")]
        assert np.all(np.diff(by_item["t_ns"].astype(np.int64)) >= 0), \
            f"copy warp {key}: items did not land in consumption order"
    return landed


def _last_landing(landed, n_counters, per_counter):
    counts = np.bincount(landed["id"].astype(np.int64), minlength=n_counters)
    assert np.array_equal(counts, np.full(n_counters, per_counter)), \
        "every counter must see its target number of landings"
    last = np.zeros(n_counters, np.int64)
    np.maximum.at(last, landed["id"].astype(np.int64), landed["t_ns"].astype(np.int64))
    return last


@pytest.mark.parametrize("S,R,K,N,c", [
    (3, 384, 512, 512, 0),     # two m-tiles per shard (the second ragged), 64 chunks per source
    (2, 256, 1024, 256, 16),
])
def test_trace_fused_f16_waits_follow_landings(S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "f16", 6100 + S + K)
    with Plan(S, S * R, K, N, "f16", c) as plan:
        ref = _run(plan, x, "f16")
        plan.set_trace(1 << 16)
        got = _run(plan, x, "f16")
        n, ev = plan.trace()
        geo = plan.geometry
        grid = plan.grid
    assert n == len(ev) > 0
    assert np.array_equal(got[0], ref[0]), "a traced run must compute the same C"
    assert np.count_nonzero(ev["kind"] == B_.TRACE_CTA_START) == grid
    assert np.count_nonzero(ev["kind"] == B_.TRACE_CTA_END) == grid
    Q, P = geo["chunks_per_source"], geo["pieces_per_chunk"]
    landed = _check_copy_order(ev)
    last = _last_landing(landed, (S - 1) * Q, P)
    ends = ev[ev["kind"] == B_.TRACE_WAIT_END]
    starts = ev[ev["kind"] == B_.TRACE_WAIT_START]
    assert len(ends) == len(starts) > 0
    for e in ends:
        pos, q0, q1 = int(e["aux"] >> 48), int((e["aux"] >> 24) & 0xFFFFFF), int(e["aux"] & 0xFFFFFF)
        assert 1 <= pos < S and 0 <= q0 <= q1 < Q
        need = last[(pos - 1) * Q + q0:(pos - 1) * Q + q1 + 1]
        assert int(e["t_ns"]) >= int(need.max()), \
            f"tile {e['id']} stopped waiting before its chunks {q0}..{q1} of position {pos} landed"
    # every remote tile waited (two CTAs of a pair: one wait each), no local tile did
    tiles = geo["tiles"]
    local_tiles = tiles // S
    assert set(ends["id"].tolist()) == set(range(local_tiles, tiles))
    done = ev[ev["kind"] == B_.TRACE_TILE_DONE]
    final = (done["aux"] & 0xFF) == (done["aux"] >> 8) - 1   # whole tiles and last parts
    assert np.count_nonzero(final) == tiles * 2
    assert sorted(set(done["id"][final].tolist())) == list(range(tiles))


@pytest.mark.parametrize("S,R,K,N", [
    (2, 32, 16384, 1024),      # the skinny workload's rows and K: 8 k-parts of 16 units
    (4, 16, 4096, 512),        # 3 remote shards, 2 k-parts
])
def test_trace_skinny_units_wait_only_for_their_part(S, R, K, N):
    x = synth.make_inputs(S, R, K, N, "i8", 6200 + S + K)
    with Plan(S, S * R, K, N, "i8") as plan:
        assert plan.path == B_.PATH_SKINNY_I8
        ref = _run(plan, x, "i8")
        plan.set_trace(1 << 18)
        got = _run(plan, x, "i8")
        n, ev = plan.trace()
        geo = plan.geometry
    assert n == len(ev) > 0
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    Q = geo["chunks_per_source"]
    landed = _check_copy_order(ev)
    per_part = (S - 1) * Q
    n_counters = int(landed["id"].max()) + 1
    assert n_counters % per_part == 0
    np_parts = n_counters // per_part
    assert np_parts > 1, "the remote rows must be released in more than one k-part"
    last = _last_landing(landed, n_counters, 1)
    ends = ev[ev["kind"] == B_.TRACE_WAIT_END]
    assert len(ends) > 0
    kq = _units_per_tile(K)
    for e in ends:
        j = int(e["aux"])
        assert j == _part_of(int(e["id"]) % kq, kq, np_parts), "a unit waits for its own k-part"
        assert int(e["t_ns"]) >= int(last[j * per_part:(j + 1) * per_part].max()), \
            f"unit {e['id']} stopped waiting before part {j} landed"
    issued = ev[ev["kind"] == B_.TRACE_UNIT_ISSUED]
    assert sorted(issued["id"].tolist()) == list(range(geo["n_tiles"] * kq))


def _units_per_tile(K):
    return ((K + 63) // 64 + 1) // 2


def _part_of(qu, kq, np_parts):
    return ((qu + 1) * np_parts + kq - 1) // kq - 1


def test_trace_skinny_missing_part_blocks_only_its_units():
    """Streaming, shown with a k-part that never lands (its copy task is skipped):
    units reading the other parts still go out; units of the missing part never
    do, and the run ends in a TIMEOUT status, not a hang."""
    S, R, K, N = 2, 32, 16384, 1024
    x = synth.make_inputs(S, R, K, N, "i8", 6250)
    kq = _units_per_tile(K)
    with Plan(S, S * R, K, N, "i8") as plan:
        ref = _run(plan, x, "i8")
        Q = plan.geometry["chunks_per_source"]
        plan.set_trace(1 << 18)
        plan.set_timeout_ns(20_000_000)
        missing = 5
        plan.set_debug(B_.DEBUG_SKIP_ITEM, missing * (S - 1) * Q)  # task (part 5, chunk 0)
        shards = [_dev(s) for s in x["shards"]]
        plan.dequant_run(shards, _dev(x["B"]), _dev(x["bias"]), _dev(x["scale"]))
        torch.cuda.synchronize()
        assert plan.status() == B_.ERR_TIMEOUT
        n, ev = plan.trace()
        landed = ev[ev["kind"] == B_.TRACE_LANDED]
        np_parts = (int(landed["id"].max()) + 1) // ((S - 1) * Q)
        assert np_parts > missing
        issued = ev[ev["kind"] == B_.TRACE_UNIT_ISSUED]
        parts = [_part_of(int(u) % kq, kq, np_parts) for u in issued["id"]]
        assert len(parts) > 0 and missing not in parts
        assert len(set(parts)) > 1
        plan.set_debug(0, 0)
        plan.set_timeout_ns(1_000_000_000)
        plan.reset()
        got = _run(plan, x, "i8")
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_trace_off_and_capacity():
    S, R, K, N = 2, 128, 256, 128
    x = synth.make_inputs(S, R, K, N, "f16", 6300)
    with Plan(S, S * R, K, N, "f16") as plan:
        with pytest.raises(B_.AgGemmError) as e:
            plan.trace()
        assert e.value.code == B_.ERR_STATE
        plan.set_trace(4)           # far too small: events are counted, at most 4 kept
        _run(plan, x, "f16")
        n, ev = plan.trace()
        assert n > 4 and len(ev) <= 4
        plan.set_trace(0)
        with pytest.raises(B_.AgGemmError):
            plan.trace()
