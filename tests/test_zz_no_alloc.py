"""The allocation-free statistics entry point (for callers that cannot call cudaMalloc, e.g.
because their device memory belongs to a pool or a host framework) must give the same results as
qwm_update_query_stats, call after call.  This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes when run alone."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from helpers import from_u16  # noqa: E402

D = 128


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_kv_cache_qsac_gb300 as qq
    return qq


def _state(H, r):
    return dict(S=torch.zeros(H, D, D, device="cuda"), n=torch.zeros(H, dtype=torch.int64, device="cuda"),
                w=torch.empty(H, D, device="cuda"), lam=torch.empty(H, D, device="cuda"),
                ur=torch.empty(H, D, r, dtype=torch.bfloat16, device="cuda"))


def _compare(q, ctx, a, b, status):
    torch.cuda.synchronize()
    assert q.qwm_sync_status(ctx) == 0 and status.item() == 0
    assert torch.equal(a["n"], b["n"])
    torch.testing.assert_close(b["S"], a["S"], rtol=1e-5, atol=1e-5 * max(float(a["S"].abs().max()), 1e-30))
    torch.testing.assert_close(b["w"], a["w"], rtol=1e-5, atol=0.0)
    la, lb = a["lam"].double(), b["lam"].double()
    assert torch.all((la - lb).abs() <= 1e-3 * la.abs() + 1e-6 * la.abs().max())
    if int(a["n"].min()) > 0:
        ua, ub = a["ur"].double(), b["ur"].double()
        cos = (ua * ub).sum(1) / (ua.norm(dim=1) * ub.norm(dim=1))
        assert torch.all(cos > 0.999), cos


def _queries(call, nq, H):
    reps = (H + 1) // 2
    return from_u16(synth.queries(synth.TINY, call, nq).repeat(reps, axis=0)[:H], torch.bfloat16)


def test_noalloc_matches_context_version_on_two_calls(q):
    H, r = 3, 8
    ctx = q.Context(heads=H, rank=r)
    a, b = _state(H, r), _state(H, r)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, nq in enumerate((256, 130)):
        qb = _queries(call, nq, H)
        q.qwm_update_query_stats(ctx, qb, nq, a["S"], a["n"], a["w"], a["lam"], a["ur"])
        q.qwm_update_query_stats_noalloc(ctx.cfg, qb, nq, b["S"], b["n"], b["w"], b["lam"], b["ur"], status)
        _compare(q, ctx, a, b, status)


@pytest.mark.parametrize("H,nqs", [(64, (300, 0)), (2, (0, 100)), (5, (100, 100))],
                         ids=["64heads_then_no_queries", "cold_then_one_short_tile", "short_tiles"])
def test_noalloc_edge_sizes(q, H, nqs):
    """The largest head count the array holds, a call with no new Queries (recompute only) and
    calls whose Queries fill less than one 128-row tile, each against the context version."""
    r = 8
    ctx = q.Context(heads=H, rank=r)
    a, b = _state(H, r), _state(H, r)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, nq in enumerate(nqs):
        qb = _queries(call, nq, H) if nq else None
        q.qwm_update_query_stats(ctx, qb, nq, a["S"], a["n"], a["w"], a["lam"], a["ur"])
        q.qwm_update_query_stats_noalloc(ctx.cfg, qb, nq, b["S"], b["n"], b["w"], b["lam"], b["ur"], status)
        _compare(q, ctx, a, b, status)


def test_noalloc_allocates_no_device_memory(q):
    """After the first call in the process (which may load the library's module, and with it the
    fixed array), further calls leave the device's free memory unchanged."""
    H, r, nq = 4, 8, 256
    b = _state(H, r)
    cfg = q.qwm_config(H, 128, 256, 64, 4, r, 2, 10, 0)
    qb = _queries(0, nq, H)
    q.qwm_update_query_stats_noalloc(cfg, qb, nq, b["S"], b["n"], b["w"], b["lam"], b["ur"])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        q.qwm_update_query_stats_noalloc(cfg, qb, nq, b["S"], b["n"], b["w"], b["lam"], b["ur"])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(b["n"][0]) == 4 * nq


def test_noalloc_rejects_more_heads_than_its_scratch(q):
    cfg = q.qwm_config(65, 128, 256, 64, 4, 8, 2, 10, 0)
    s = _state(65, 8)
    with pytest.raises(q.QwmError) as e:
        q.qwm_update_query_stats_noalloc(cfg, None, 0, s["S"], s["n"], s["w"], s["lam"], s["ur"])
    assert e.value.status == q.QWM_ERR_SHAPE
