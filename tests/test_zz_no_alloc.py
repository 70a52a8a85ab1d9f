"""The allocation-free permutation gives the same results as moe_permute.

moe_permute_noalloc exists for callers that cannot allocate device memory (for example code
running under stream capture or inside a runtime's enqueue callback) and so cannot pass a
workspace.  It keeps its scratch in a fixed array inside the library, shared by every call;
two calls in a row must each match moe_permute exactly, so nothing left in the array by the
first call may leak into the second.  This file is collected last on purpose."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_56_b300 as m
    m._native.lib()
    return m


def _both(moe, idx_np, n):
    T, k = idx_np.shape
    ti = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    ws = moe.workspace(max(T, 1), 64, 64, n, k, torch.bfloat16, DEV)
    ref = moe.moe_permute(ti, n, ws)
    assert moe.moe_check_device_error(ws) == 0
    out = (torch.full((n + 1,), -7, dtype=torch.int32, device=DEV),
           torch.full((T * k,), -7, dtype=torch.int32, device=DEV),
           torch.full((T * k,), -7, dtype=torch.int32, device=DEV))
    moe.moe_permute_noalloc(ti, n, expert_offsets=out[0], perm=out[1], inv_perm=out[2])
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)


def test_permute_noalloc_matches_permute_on_two_calls_in_a_row(moe):
    rng = np.random.default_rng(11)
    # multi-block (per-block counts in the fixed array), then a differently routed
    # multi-block batch with other block counts, then a single-block batch
    first = rng.integers(0, 8, size=(150001, 2))
    second = np.minimum(rng.geometric(0.35, size=(90000, 2)) - 1, 7)
    _both(moe, first, 8)
    _both(moe, second, 8)
    _both(moe, rng.integers(0, 32, size=(1000, 2)), 32)


def test_permute_noalloc_rejects_sizes_beyond_its_array(moe):
    from sparse_mixture_experts_56_b300 import _native
    fake = 4096  # never dereferenced: the size check fails first
    st = _native.lib().moe_permute_noalloc(fake, 2_100_000, 2, 8, fake, fake, fake, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
