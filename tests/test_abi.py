"""C-ABI library checks that need no GPU: it loads, exports every function the
header declares, and rejects host-checkable bad arguments before touching CUDA."""
import ctypes

import pytest

import __graft_entry__


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    from speculative_decoding_verification_15_gb300 import binding

    return binding.load()


def test_exports_every_header_function(lib):
    from speculative_decoding_verification_15_gb300 import binding

    names = binding.header_functions()
    assert {"spec_verify_greedy", "spec_verify_sample", "spec_schedule_verify_len",
            "spec_verify_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_binding_has_same_names():
    import speculative_decoding_verification_15_gb300 as pkg

    for n in ("spec_verify_greedy", "spec_verify_sample", "spec_schedule_verify_len",
              "spec_verify_workspace_size"):
        assert callable(getattr(pkg, n))


def _sample(lib, **kw):
    a = dict(target=ctypes.c_void_p(16), draft=ctypes.c_void_p(16), dtype=0, B=2, Kmax=3, V=100, ld=100,
             x=ctypes.c_void_p(16), nd=None, T=ctypes.c_void_p(16), seed=0, step=0,
             tok=ctypes.c_void_p(16), acc=ctypes.c_void_p(16), p=None, q=None, st=ctypes.c_void_p(16),
             ws=ctypes.c_void_p(16), wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.spec_verify_sample(a["target"], a["draft"], a["dtype"], a["B"], a["Kmax"], a["V"], a["ld"],
                                  a["x"], a["nd"], a["T"], a["seed"], a["step"], a["tok"], a["acc"], a["p"],
                                  a["q"], a["st"], a["ws"], a["wsb"], a["stream"])


def test_host_argument_errors(lib):
    EINVAL, EUNSUP = 1, 3
    assert _sample(lib, B=0) == 0                 # empty batch: no-op
    assert _sample(lib, B=-1) == EINVAL
    assert _sample(lib, V=0) == EINVAL
    assert _sample(lib, ld=99) == EINVAL          # ld_row < V
    assert _sample(lib, dtype=7) == EINVAL
    assert _sample(lib, target=None) == EINVAL
    assert _sample(lib, T=None) == EINVAL
    assert _sample(lib, draft=None) == EINVAL
    assert _sample(lib, x=None) == EINVAL
    assert _sample(lib, st=None) == EINVAL
    assert _sample(lib, Kmax=256) == EUNSUP
    assert _sample(lib, B=8193) == EUNSUP
    g = lib.spec_verify_greedy(None, 0, 1, 1, 10, 10, None, None, None, None, None, None, 0, None)
    assert g == EINVAL
    assert lib.spec_verify_greedy(None, 0, 0, 1, 10, 10, None, None, None, None, None, None, 0, None) == 0


def test_scheduler_host_argument_errors(lib):
    EINVAL, EUNSUP = 1, 3
    P = ctypes.c_void_p(16)
    # budget below B * min_len
    assert lib.spec_schedule_verify_len(P, None, 4, 4, P, 100, 3, 1, P, None, None) == EINVAL
    # table too short for the mandatory slots
    assert lib.spec_schedule_verify_len(P, None, 4, 4, P, 4, 100, 1, P, None, None) == EINVAL
    assert lib.spec_schedule_verify_len(P, None, 4, 4, None, 100, 100, 1, P, None, None) == EINVAL
    assert lib.spec_schedule_verify_len(P, None, 1025, 8, P, 10000, 9000, 0, P, None, None) == EUNSUP


def test_error_strings(lib):
    assert lib.spec_error_string(0) == b"ok"
    assert b"workspace" in lib.spec_error_string(4)


def test_early_exit_host_argument_errors(lib):
    """The early-exit calls check their arguments as the two-kernel calls do."""
    EINVAL, EUNSUP = 1, 3
    P = ctypes.c_void_p(16)

    def ee(**kw):
        a = dict(target=P, draft=P, dtype=0, B=2, Kmax=3, V=100, ld=100, x=P, nd=None, T=P, tok=P, acc=P, st=P)
        a.update(kw)
        return lib.spec_verify_sample_early_exit(a["target"], a["draft"], a["dtype"], a["B"], a["Kmax"], a["V"],
                                                 a["ld"], a["x"], a["nd"], a["T"], 0, 0, a["tok"], a["acc"], None,
                                                 None, a["st"], None)

    assert ee(B=0) == 0
    assert ee(B=-1) == EINVAL and ee(V=0) == EINVAL and ee(ld=99) == EINVAL and ee(dtype=2) == EINVAL
    assert ee(Kmax=256) == EUNSUP and ee(B=8193) == EUNSUP
    assert ee(target=None) == EINVAL and ee(tok=None) == EINVAL and ee(st=None) == EINVAL
    assert ee(x=None) == EINVAL and ee(T=None) == EINVAL and ee(draft=None) == EINVAL
    assert ee(target=ctypes.c_void_p(17)) == EINVAL  # bf16 rows need 2-byte alignment
    assert lib.spec_verify_greedy_early_exit(None, 0, 1, 1, 10, 10, P, None, P, P, P, None) == EINVAL
    assert lib.spec_verify_greedy_early_exit(P, 0, 0, 1, 10, 10, None, None, None, None, None, None) == 0


def test_flat_host_argument_errors(lib):
    EINVAL = 1
    P = ctypes.c_void_p(16)
    # no offsets
    assert lib.spec_verify_greedy_flat(P, 0, 2, 3, 100, 100, None, P, P, P, P, P, 1 << 30, None) == EINVAL
    assert lib.spec_verify_sample_flat(P, P, 0, 2, 3, 100, 100, None, P, P, 0, 0, P, P, None, None, P, P, 1 << 30,
                                       None) == EINVAL
    assert lib.spec_verify_greedy_flat(P, 0, 0, 3, 100, 100, None, None, None, None, None, None, 0, None) == 0


def test_markov_host_argument_errors(lib):
    """spec_markov_draft rejects bad sizes, ranks, pointers and alignment before any launch."""
    EINVAL, EUNSUP = 1, 3
    P = ctypes.c_void_p(16)

    def mk(**kw):
        a = dict(base=P, dtype=0, B=2, K=3, V=100, ld=100, anchor=P, emb=P, proj=P, r=8, T=P, tok=P, z=P, st=P)
        a.update(kw)
        return lib.spec_markov_draft(a["base"], a["dtype"], a["B"], a["K"], a["V"], a["ld"], a["anchor"], a["emb"],
                                     a["proj"], a["r"], a["T"], 0, 0, a["tok"], a["z"], a["st"], None)

    assert mk(B=0) == 0
    assert mk(B=-1) == EINVAL and mk(K=-1) == EINVAL and mk(V=0) == EINVAL and mk(ld=99) == EINVAL
    assert mk(r=0) == EINVAL and mk(dtype=5) == EINVAL
    assert mk(r=513) == EUNSUP and mk(r=6) == EUNSUP  # at most 512, a multiple of 4
    assert mk(B=8193) == EUNSUP and mk(K=256) == EUNSUP
    assert mk(anchor=None) == EINVAL and mk(emb=None) == EINVAL and mk(proj=None) == EINVAL
    assert mk(st=None) == EINVAL and mk(base=None) == EINVAL and mk(tok=None) == EINVAL and mk(z=None) == EINVAL
    assert mk(emb=ctypes.c_void_p(17)) == EINVAL and mk(z=ctypes.c_void_p(18)) == EINVAL


def test_markov_topk_host_argument_errors(lib):
    """spec_markov_draft_topk: the candidate count, the workspace and the checks of
    spec_markov_draft, before any launch; the workspace is B K min(topk, V) int32."""
    EINVAL, EUNSUP, EWS = 1, 3, 4
    P = ctypes.c_void_p(16)
    ws_size = lib.spec_markov_topk_workspace_size
    assert ws_size(64, 7, 151936, 64) == 64 * 7 * 64 * 4
    assert ws_size(3, 2, 10, 64) == 256  # min(topk, V) = 10 candidates, 240 bytes rounded up to 256
    assert ws_size(1, 1, 10, 0) == 0 and ws_size(1, 1, 10, 1025) == 0 and ws_size(-1, 1, 10, 4) == 0

    def mk(**kw):
        a = dict(base=P, dtype=0, B=2, K=3, V=100, ld=100, anchor=P, emb=P, proj=P, r=8, T=P, topk=16, tok=P, z=P,
                 st=P, ws=P, wsb=1 << 20)
        a.update(kw)
        return lib.spec_markov_draft_topk(a["base"], a["dtype"], a["B"], a["K"], a["V"], a["ld"], a["anchor"],
                                          a["emb"], a["proj"], a["r"], a["T"], 0, 0, a["topk"], a["tok"], a["z"],
                                          a["st"], a["ws"], a["wsb"], None)

    assert mk(B=0) == 0
    assert mk(topk=0) == EINVAL and mk(topk=-3) == EINVAL and mk(topk=1025) == EUNSUP
    assert mk(B=-1) == EINVAL and mk(V=0) == EINVAL and mk(ld=99) == EINVAL and mk(r=6) == EUNSUP
    assert mk(anchor=None) == EINVAL and mk(tok=None) == EINVAL and mk(st=None) == EINVAL
    assert mk(ws=None) == EWS and mk(wsb=2 * 3 * 16 * 4 - 1) == EWS and mk(ws=ctypes.c_void_p(24)) == EWS
    assert mk(z=ctypes.c_void_p(18)) == EINVAL


def test_threshold_host_argument_errors(lib):
    EINVAL = 1
    P = ctypes.c_void_p(16)
    assert lib.spec_schedule_threshold(P, None, 4, 4, ctypes.c_float(float("nan")), P, None) == EINVAL
    assert lib.spec_schedule_threshold(None, None, 4, 4, ctypes.c_float(0.5), P, None) == EINVAL
    assert lib.spec_schedule_threshold(P, None, 0, 4, ctypes.c_float(0.5), None, None) == 0


def _ws_formula(B, K, V, esz):
    """The workspace size the header states for spec_verify_workspace_size."""
    max_e = 65504 // esz
    cpr = -(-V // max_e)
    ce = (-(-V // cpr) + 7) & ~7
    cpr = -(-V // ce)
    P = -(-(-(-V // 1024)) // 8)

    def a256(x):
        return (x + 255) & ~255

    return (256 + a256(4 * (B + 1)) + a256(128 * B) + a256(16 * B * 2 * K * cpr) + a256(32 * B * 2 * K * cpr)
            + a256(16 * B * P))


def test_workspace_size_formula(lib):
    """spec_verify_workspace_size needs no GPU and follows the header's formula."""
    for B, K, V in ((1, 0, 1), (1, 4, 1024), (64, 7, 151936), (8, 8, 32000), (256, 16, 129280), (512, 4, 151936),
                    (8192, 255, 97), (3, 255, 1 << 20)):
        for dt, esz in ((0, 2), (1, 4)):
            assert lib.spec_verify_workspace_size(B, K, V, dt) == _ws_formula(B, K, V, esz), (B, K, V, dt)
    assert lib.spec_verify_workspace_size(8193, 1, 10, 0) == 0 and lib.spec_verify_workspace_size(1, 256, 10, 0) == 0


def test_fixed_scratch_limits_stated_in_the_header(lib):
    """The batch sizes the header gives for spec_verify_sample_noalloc at V = 151936,
    Kmax = 7: the largest B whose workspace fits SPEC_STATIC_SCRATCH_BYTES (4 MiB)."""
    scratch = 4 << 20
    for dt, bmax in ((0, 1104), (1, 586)):
        assert lib.spec_verify_workspace_size(bmax, 7, 151936, dt) <= scratch
        assert lib.spec_verify_workspace_size(bmax + 1, 7, 151936, dt) > scratch
