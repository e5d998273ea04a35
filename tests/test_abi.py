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
