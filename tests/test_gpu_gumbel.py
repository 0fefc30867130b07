"""GPU test of the Gumbel noise the temperature walks add for the bonus draw
(ddtree_testing_gumbel, include/ddtree_testing.h), over every value of U.

U = ((w >> 8) + 0.5) 2^-24 takes 2^24 values, so the check is exhaustive: the
fp32 noise must lie within 2e-6 of -log(-log U) computed in fp64 (with
-log U = -log1p(-(1 - U)) and 1 - U exact above one half). A bonus draw whose
two best perturbed scores differ by more than the parity bar's margin cannot
change by that much, so the walks' decisions stay those of the fp64 oracle.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402


def test_gumbel_noise_every_uniform():
    lib = dd.load_library()
    fn = lib.ddtree_testing_gumbel
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    n = 1 << 24
    k = np.arange(n, dtype=np.uint32)
    low = np.random.default_rng(3).integers(0, 256, size=n, dtype=np.uint32)   # ignored bits
    words = torch.from_numpy(((k << np.uint32(8)) | low).view(np.int32)).cuda()
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    assert fn(words.data_ptr(), out.data_ptr(), n, None) == 0
    torch.cuda.synchronize()
    g = out.cpu().numpy().astype(np.float64)
    kd = k.astype(np.float64)
    u = (kd + 0.5) * 2.0 ** -24
    one_minus_u = ((2.0 ** 24 - 1.0 - kd) + 0.5) * 2.0 ** -24
    e = np.where(u < 0.5, -np.log(u), -np.log1p(-one_minus_u))
    err = np.abs(g - (-np.log(e)))
    assert np.all(np.isfinite(g))
    assert err.max() < 2e-6, (float(err.max()), int(np.argmax(err)))

