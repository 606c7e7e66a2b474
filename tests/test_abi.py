"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol that include/*.h declare, and validates configurations before touching CUDA."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    return sorted(set(re.findall(r"QWM_API\s+[\w\s\*]*?\b(qwm_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def qwm():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_kv_cache_qsac_gb300 as q
    return q


def test_header_declares_the_five_path_calls():
    decl = _declared()
    for name in ("qwm_update_query_stats", "qwm_fit_centroids", "qwm_quantize_kv", "qwm_attend",
                 "qwm_dequantize", "qwm_create", "qwm_destroy", "qwm_sync_status"):
        assert name in decl


def test_library_exports_every_declared_symbol(qwm):
    lib = qwm.raw_library()
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(qwm.EXPORTED)


def test_config_validation(qwm):
    good = qwm.qwm_config(40, 128, 256, 64, 4, 8, 2, 10, 0)
    assert qwm.qwm_workspace_bytes(good) > 0
    for bad in (qwm.qwm_config(40, 96, 256, 64, 4, 8, 2, 10, 0),     # head_dim
                qwm.qwm_config(40, 128, 100, 64, 4, 8, 2, 10, 0),    # centroids
                qwm.qwm_config(40, 128, 256, 32, 4, 8, 2, 10, 0),    # group
                qwm.qwm_config(40, 128, 256, 64, 17, 8, 2, 10, 0),   # top_m
                qwm.qwm_config(40, 128, 256, 64, 4, 17, 2, 10, 0),   # rank
                qwm.qwm_config(40, 128, 256, 64, 4, 8, 3, 10, 0),    # bits
                qwm.qwm_config(0, 128, 256, 64, 4, 8, 2, 10, 0)):    # heads
        assert qwm.qwm_workspace_bytes(bad) == 0
        h = C.c_void_p()
        st = qwm.raw_library().qwm_create(C.byref(bad), C.byref(h))
        assert st in (qwm.QWM_ERR_ARG, qwm.QWM_ERR_SHAPE, qwm.QWM_ERR_UNSUPPORTED) and not h.value


def test_null_arguments_rejected_before_cuda(qwm):
    lib = qwm.raw_library()
    assert lib.qwm_create(None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_destroy(None) == qwm.QWM_ERR_ARG
    assert lib.qwm_update_query_stats(None, None, 0, None, None, None, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_fit_centroids(None, None, 0, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_fit_centroids_kv(None, None, None, 0, None, None, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_quantize_kv(None, None, None, 0, None, None, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_attend(None, None, 0, None, 0, 1.0, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_attend_merge(None, None, 0, None, 0, 1.0, None, None, 0, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_dequantize(None, None, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_sync_status(None, None) == qwm.QWM_ERR_ARG
    assert qwm.qwm_status_string(qwm.QWM_ERR_NOT_CONVERGED).startswith("eigensolver")


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The CUDA package neither imports the oracle nor carries a CPU implementation."""
    pkg = os.path.join(ROOT, "bit_kv_cache_qsac_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "liboracle" not in txt, f


def test_new_calls_reject_null_arguments(qwm):
    lib = qwm.raw_library()
    assert lib.qwm_dequantize_chunks(None, None, 0, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_select_rank(None, None, 0.5, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_psac_kept(None, None, None, None) == qwm.QWM_ERR_ARG
    assert lib.qwm_psac_pack(None, None, None, None, None, None, None, None) == qwm.QWM_ERR_ARG
    bad = qwm.qwm_config(4, 128, 256, 64, 4, 8, 2, 10, 0, 0, 0, 2)     # an unknown test flag
    assert qwm.qwm_workspace_bytes(bad) == 0


def test_psac_plan_matches_the_oracle_rule(qwm):
    """The per-head layout plan (host only): each head the smaller of dense and sparse, laid out one
    after the other, as the oracle's byte-count rule chooses."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(5)
    for n in (1, 127, 128, 4680, 10800):
        H = 40
        cfg = qwm.qwm_config(H, 128, 256, 64, 4, 16, 2, 10, 0)
        ranks = rng.integers(0, 17, H)
        kept = rng.integers(0, n + 1, H)
        plan, c_bytes, n_scales, _ = qwm.qwm_psac_plan(cfg, n, ranks, kept)
        want = oracle.psac_plan(n, ranks, kept)
        off_c = off_s = 0
        for h in range(H):
            c_off, s_off, r, sparse = plan[h]
            assert (bool(sparse), r) == (want[h][0], int(ranks[h]))
            assert (c_off, s_off) == (off_c, off_s)
            off_c += want[h][1] * int(ranks[h])
            off_s += want[h][1]
        assert (c_bytes, n_scales) == (off_c, off_s)
    with pytest.raises(qwm.QwmError):
        qwm.qwm_psac_plan(qwm.qwm_config(2, 128, 256, 64, 4, 8, 2, 10, 0), 100, [9, 1], [5, 5])   # rank > config
