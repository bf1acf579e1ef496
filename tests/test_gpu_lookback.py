"""The radix sort's one bounded device wait, made to run out: the decoupled look-back of
a one-sweep pass gives up after its poll limit when an earlier tile never publishes its
counts, flags the error, and the call returns GS_ERR_TIMEOUT instead of hanging.  The
kernel is the product's, unmodified: a test-only launcher starts its ticket counter at 1,
so the first block to run waits on tile 0, which no block takes.  Nothing faults: every
access stays inside the buffers, and the context stays usable (a full gs_bin_sort on the
radix path runs correctly afterwards)."""

import ctypes as C

import numpy as np
import pytest

GS_ERR_TIMEOUT = 4


@pytest.mark.gpu
def test_lookback_wait_gives_up_and_reports_a_timeout():
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    lib = gs.library()
    lib.gs_test_lookback_timeout_ws_bytes.restype = C.c_size_t
    lib.gs_test_lookback_timeout_ws_bytes.argtypes = [C.c_int64]
    lib.gs_test_lookback_timeout.restype = C.c_int
    lib.gs_test_lookback_timeout.argtypes = [C.c_void_p] * 4 + [C.c_int64, C.c_void_p,
                                                                C.c_size_t, C.c_void_p]
    n = 8192  # two 4096-key tiles
    keys = torch.randint(0, 1 << 20, (n,), dtype=torch.int32, device="cuda")
    vals = torch.arange(n, dtype=torch.int32, device="cuda")
    kout = torch.empty_like(keys)
    vout = torch.empty_like(vals)
    nb = lib.gs_test_lookback_timeout_ws_bytes(n)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    status = lib.gs_test_lookback_timeout(keys.data_ptr(), vals.data_ptr(), kout.data_ptr(),
                                          vout.data_ptr(), n, ws.data_ptr(), nb, st)
    assert status == GS_ERR_TIMEOUT
    torch.cuda.synchronize()
    # the context is intact: the same kind of sort, run for real, is still exact
    from gpu_util import check_binning, run_forward
    import oracle
    import synthetic_scenes as ss

    rng = np.random.default_rng(2)
    sc, cam = ss.random_scene(rng, 3000, 200, 120, sh_degree=1, log_scale=(-2.8, 0.8))
    g = run_forward(sc, cam, capacity=8 << 20)
    ref = oracle.render(sc, cam)
    check_binning(g, ref.binning)


def test_lookback_test_hook_rejects_bad_sizes():
    from differentiable_gaussian_splatting_gb300 import build

    build.build()
    import differentiable_gaussian_splatting_gb300 as gs

    lib = gs.library()
    lib.gs_test_lookback_timeout.restype = C.c_int
    lib.gs_test_lookback_timeout.argtypes = [C.c_void_p] * 4 + [C.c_int64, C.c_void_p,
                                                                C.c_size_t, C.c_void_p]
    fake = C.c_void_p(0x100000)  # never dereferenced: the checks fail first
    assert lib.gs_test_lookback_timeout(fake, fake, fake, fake, 4096, fake, 1 << 20, None) == 1
    assert lib.gs_test_lookback_timeout(fake, fake, fake, fake, 8192, fake, 16, None) == 5
