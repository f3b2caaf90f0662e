"""Per-kernel parity on the GPU through the C ABI: the projection kernels (W4A16 dequant GEMV
and bf16 GEMV) and the greedy argmax, against the CPU oracle's definitions."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


def _linear(fmt, n_out, n_in, seed):
    cfg = dict(synth.get_config("tiny"))
    rng_cfg = synth.weights
    with rng_cfg._pool() as pool:
        if fmt == "bf16":
            return {"w": rng_cfg._normal_bf16((n_out, n_in), 0.02, seed, 77, pool), "shape": (n_out, n_in)}
        return rng_cfg._int4_linear(n_out, n_in, 0.004, seed, 77, pool)


def _dense(fmt, lin):
    if fmt == "bf16":
        return oracle.bf16_bits_to_float(lin["w"], np.float64)
    return oracle.dequant_w4a16(lin["packed"], lin["scales"], np.float64)


SHAPES = [(32, 32), (40, 64), (96, 288), (256, 1536), (2560, 1536), (1536, 2048), (1536, 4096),
          (512, 256), (1536, 256), (1536, 6144), (1536, 12288), (8960, 1536), (12288, 1536)]


@pytest.mark.parametrize("fmt", ["bf16", "w4a16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_linear_matches_oracle(rt, fmt, shape):
    n_out, n_in = shape
    lin = _linear(fmt, n_out, n_in, seed=n_out * 7 + n_in)
    W = _dense(fmt, lin)
    op = rt.LinearOp(fmt, lin)
    rng = np.random.default_rng(n_out + n_in)
    for nb in (1, 2, 3, 4):  # the GEMV (5 rows and up take the tensor-core path)
        x = rng.standard_normal((nb, n_in)).astype(np.float32)
        y = op(torch.from_numpy(x).cuda()).cpu().numpy()
        ref = x.astype(np.float64) @ W.T
        bound = 1e-5 * (np.abs(x).astype(np.float64) @ np.abs(W).T) + 1e-7
        assert np.all(np.abs(y - ref) <= bound), (fmt, shape, nb, np.max(np.abs(y - ref) / bound))
        np.testing.assert_allclose(y, ref, rtol=1e-2, atol=1e-4 * np.max(np.abs(ref)))
    op.close()


def test_int4_exact_with_integer_activations(rt):
    """Hand-built int4 rows, power-of-two scales and integer activations: every product and
    partial sum is exact in fp32, so the kernel must reproduce the result bit for bit.  This
    pins nibble order, sign handling and the repack."""
    n_out, n_in = 64, 512
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, (n_out, n_in))
    q[0, :16] = np.arange(-8, 8)
    nib = (q.reshape(n_out, n_in // 8, 8) & 0xF).astype(np.uint32)
    packed = np.bitwise_or.reduce(nib << (np.arange(8, dtype=np.uint32) * 4), axis=2).view(np.int32)
    exps = rng.integers(-3, 3, (n_out, n_in // 32))
    scales = (np.array(2.0, np.float32) ** exps).astype(np.float32).view(np.uint32) >> 16
    lin = {"packed": packed, "scales": scales.astype(np.uint16), "shape": (n_out, n_in)}
    op = rt.LinearOp("w4a16", lin)
    x = rng.integers(-4, 5, (3, n_in)).astype(np.float32)
    y = op(torch.from_numpy(x).cuda()).cpu().numpy()
    W = q * np.repeat(2.0 ** exps, 32, axis=1)
    np.testing.assert_array_equal(y, (x.astype(np.float64) @ W.T).astype(np.float32))
    op.close()


def test_int4_bf16_rounding_of_products(rt):
    """bf16(q * s) at round-to-nearest-even ties, read through one-hot activations."""
    cases = [(3, 1 + 1 / 128), (3, 1 + 3 / 128), (5, 1 + 1 / 128), (-3, 1 + 3 / 128), (7, 1 + 127 / 128),
             (-8, 1.5), (-7, 1 + 5 / 128), (6, 1 + 101 / 128)]
    n_in = 32 * len(cases)
    q = np.zeros((32, n_in), int)
    s = np.zeros((32, len(cases)), np.float32)
    for g, (qq, ss) in enumerate(cases):
        q[:, 32 * g:32 * (g + 1)] = qq
        s[:, g] = ss
    nib = (q.reshape(32, n_in // 8, 8) & 0xF).astype(np.uint32)
    packed = np.bitwise_or.reduce(nib << (np.arange(8, dtype=np.uint32) * 4), axis=2).view(np.int32)
    scales = (s.view(np.uint32) >> 16).astype(np.uint16)
    lin = {"packed": packed, "scales": scales, "shape": (32, n_in)}
    op = rt.LinearOp("w4a16", lin)
    x = np.zeros((len(cases), n_in), np.float32)
    for g in range(len(cases)):
        x[g, 32 * g + 5] = 1.0
    y = op(torch.from_numpy(x).cuda()).cpu().numpy()
    W = oracle.dequant_w4a16(packed, scales)
    for g in range(len(cases)):
        assert np.all(y[g] == W[:, 32 * g + 5]), (cases[g], y[g][0], W[0, 32 * g + 5])
    op.close()


def test_argmax_rows_planted_ties(rt):
    rng = np.random.default_rng(5)
    n, V = 6, 262144
    x = rng.standard_normal((n, V)).astype(np.float32)
    x[0, [7, 4095, 4096, 200000]] = 50.0          # ties across block boundaries -> 7
    x[1, [V - 1, 131072]] = 60.0                   # -> 131072
    x[2, :] = 1.0                                  # all equal -> 0
    x[3, [10, 20]] = np.inf                        # inf ties -> 10
    x[4, :100] = -np.inf
    x[5, [99999]] = 7.0
    ids = rt.argmax_rows(torch.from_numpy(x).cuda()).cpu().numpy()
    assert ids.tolist() == oracle.greedy_argmax(x).tolist() == [7, 131072, 0, 10, int(np.argmax(x[4])), 99999]


def test_argmax_rows_ignores_nan(rt):
    x = np.zeros((1, 5000), np.float32)
    x[0, 3] = np.nan
    x[0, 4100] = 2.0
    x[0, 17] = 2.0
    assert rt.argmax_rows(torch.from_numpy(x).cuda()).cpu().numpy().tolist() == [17]


@pytest.mark.parametrize("fmt", ["bf16", "w4a16"])
@pytest.mark.parametrize("shape", [(128, 64), (96, 288), (2560, 1536), (1536, 2048), (1536, 6144),
                                   (8960, 1536), (12288, 1536), (1536, 256), (256, 1536)])
def test_linear_tensor_core_batches(rt, fmt, shape):
    """Batches >= 5 run the tcgen05 dequant GEMM (bf16 x_hi + x_lo against bf16(q*s), fp32
    accumulation in TMEM); it must match the oracle's dense product like the GEMV does."""
    n_out, n_in = shape
    lin = _linear(fmt, n_out, n_in, seed=n_out * 3 + n_in)
    W = _dense(fmt, lin)
    op = rt.LinearOp(fmt, lin)
    rng = np.random.default_rng(abs(n_out - n_in))
    for nb in (5, 16, 17, 40, 64):
        x = rng.standard_normal((nb, n_in)).astype(np.float32)
        y = op(torch.from_numpy(x).cuda()).cpu().numpy()
        ref = x.astype(np.float64) @ W.T
        # x_lo leaves |x| * 2^-17 per element; fp32 accumulation adds the rest
        bound = 4e-5 * (np.abs(x).astype(np.float64) @ np.abs(W).T) + 1e-6
        assert np.all(np.abs(y - ref) <= bound), (fmt, shape, nb, np.max(np.abs(y - ref) / bound))
        np.testing.assert_allclose(y, ref, rtol=1e-2, atol=1e-4 * np.max(np.abs(ref)))
    op.close()
