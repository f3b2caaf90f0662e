"""The allocation-free argmax entry point (g4_argmax_rows_static) against the allocating one.

Collected last on purpose: it reuses one fixed scratch array inside the library, so it runs
after every other test, and it must also pass alone in a fresh process.  Two calls in a row
check that the array's leftover contents from the first call do not leak into the second."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


def test_static_argmax_matches_allocating_entry_point(rt):
    rng = np.random.default_rng(17)
    first = rng.standard_normal((64, 262144)).astype(np.float32)
    first[3, [5, 70000]] = 9.0                  # a tie: the lower index wins
    second = rng.standard_normal((7, 100001)).astype(np.float32)
    second[1, :] = 0.5
    for x in (first, second):                   # two calls in a row share the scratch
        d = torch.from_numpy(x).cuda()
        got = rt.argmax_rows_static(d).cpu().numpy()
        want = rt.argmax_rows(d).cpu().numpy()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got, want)
        np.testing.assert_array_equal(got, np.argmax(x, axis=1))


def test_static_argmax_rejects_sizes_beyond_its_scratch(rt):
    from accelerator_decode_gb300 import g4
    with pytest.raises(g4.G4Error) as e:
        rt.argmax_rows_static(torch.zeros(65, 8, device="cuda"))
    assert e.value.status == g4.G4_ERR_INVALID_ARG
    with pytest.raises(g4.G4Error):
        rt.argmax_rows_static(torch.zeros(1, 1048577, device="cuda"))
