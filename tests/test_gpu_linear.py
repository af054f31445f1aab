"""The FP8 linear layer with a per-group FP8 output, on the GPU through the C
ABI, against the oracle.

COAT review page, section 3: linear layers take per-tensor FP8 inputs
("mixed-granularity activation quantization"), and the GEMM's epilogue
quantizes its output tile per 1 x G group ("Triton kernels", linear layer
optimisation).

The kernel runs on the fifth-generation tensor cores (CTA pairs sharing one
MMA, TMA-fed shared-memory rings, accumulators in tensor memory) and
accumulates in float32, so its y is not the oracle's correctly rounded one;
the checks are
  * y within the float32 summation bound (K + 2) 2^-24 |sx sw| sum_k |x_k w_k|
    of the oracle's y (K - 1 additions, the product by RN(sx sw) and that
    rounding itself, each at most half an ulp of a partial sum);
  * (q, scale) bit-identical to the oracle's absmax quantizer applied to the
    kernel's own y: the epilogue's quantization is exact;
  * against the oracle's (q, scale): codes within one E4M3 step and scales
    within the bound above carried through max|y| / 448.
"""
import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _gpu(xq, sx, wq, sw, G, want_y=True):
    M, K = xq.shape
    N = wq.shape[0]
    dx = torch.from_numpy(np.ascontiguousarray(xq)).cuda()
    dw = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    q = torch.full((M, N), 0xAA, dtype=torch.uint8, device="cuda")
    S = torch.full((M, N // G), -1.0, dtype=torch.float32, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") if want_y else None
    coat.coat_fp8_linear_group_quantize(dx, sx, dw, sw, G, q, S, y)
    torch.cuda.synchronize()
    assert coat.coat_kernel_wait_timeouts(reset=True) == 0, "a pipeline wait gave up"
    return (y.cpu().numpy() if want_y else None), q.cpu().numpy(), S.cpu().numpy()


def _abs_products(xq, wq):
    dec = np.abs(oracle.e4m3_decode_all())
    return dec[xq] @ dec[wq].T


def _check(xq, sx, wq, sw, G, y, q, S, rows=None):
    """All three checks on the rows `rows` of the output (all by default)."""
    K = xq.shape[1]
    xs = xq if rows is None else xq[rows]
    yo, qo, So = oracle.linear_group_quantize(xs, sx, wq, sw, G)
    bound = (K + 2) * 2.0 ** -24 * (float(np.float32(sx)) * float(np.float32(sw))) * _abs_products(xs, wq)
    err = np.abs(y.astype(np.float64) - yo.astype(np.float64))
    worst = float((err / np.maximum(bound, 1e-300)).max())
    assert (err <= bound).all(), f"y outside the fp32 summation bound (worst {worst:.3f} of it)"
    # the epilogue's quantization of the kernel's own y is exact
    qk, Sk = oracle.absmax_quantize(y, G)
    assert np.array_equal(S.ravel().view(np.uint32), Sk.view(np.uint32)), "scales of y"
    bad = np.nonzero(q.ravel() != qk)[0]
    assert bad.size == 0, "codes of y: " + "; ".join(
        f"[{i}] y={float(y.ravel()[i])!r} S={float(S.ravel()[i // G])!r} "
        f"kernel {int(q.ravel()[i]):#04x} oracle {int(qk[i]):#04x}" for i in bad[:6])
    # and against the oracle's output
    gmax = bound.reshape(bound.shape[0], -1, G).max(axis=2) / 448.0
    sd = np.abs(S.astype(np.float64) - So.astype(np.float64))
    assert (sd <= gmax * (1 + 1e-6) + np.spacing(So) ).all(), "scales vs the oracle"
    P.compare_codes(q.ravel(), qo.ravel(), f"q G={G}")
    return worst


@pytest.mark.parametrize("G", [8, 16, 32, 64, 128])
def test_matches_oracle_over_several_tiles(G):
    M, N, K = 256, 384, 320          # 2 x 3 CTA tiles, 5 K steps
    xq = synth.fp8_operand_codes_np(M, K, 1 + G)
    wq = synth.fp8_operand_codes_np(N, K, 2 + G)
    sx, sw = 0.0123, 0.0371
    y, q, S = _gpu(xq, sx, wq, sw, G)
    worst = _check(xq, sx, wq, sw, G, y, q, S)
    print(f"G={G}: worst |dy| = {worst:.3f} of the summation bound")


@pytest.mark.parametrize("M,N,K,G", [(200, 272, 208, 16), (1, 16, 16, 16), (37, 48, 48, 8),
                                     (129, 2064, 1040, 16), (300, 384, 4112, 128)])
def test_ragged_shapes(M, N, K, G):
    """Sizes that are not multiples of the 128 x 256 x 128 tiles: the loads
    beyond the edges read zeros and the stores beyond them are skipped."""
    xq = synth.fp8_operand_codes_np(M, K, M + 1)
    wq = synth.fp8_operand_codes_np(N, K, N + 2)
    y, q, S = _gpu(xq, 0.0173, wq, 0.0291, G)
    _check(xq, 0.0173, wq, 0.0291, G, y, q, S)


def test_more_tiles_than_sms():
    """160 tiles of 256 x 256: each persistent CTA pair takes two or more,
    alternating between its two tensor-memory accumulators."""
    M, N, K, G = 256 * 20, 256 * 8, 256, 32
    xq = synth.fp8_operand_codes_np(M, K, 31)
    wq = synth.fp8_operand_codes_np(N, K, 32)
    y, q, S = _gpu(xq, 0.031, wq, 0.0047, G)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))
    _check(xq, 0.031, wq, 0.0047, G, y[rows], q[rows], S[rows], rows=rows)


def test_without_y_gives_the_same_codes():
    M, N, K, G = 128, 256, 192, 16
    xq = synth.fp8_operand_codes_np(M, K, 5)
    wq = synth.fp8_operand_codes_np(N, K, 6)
    y, q, S = _gpu(xq, 0.5, wq, 0.25, G)
    _, q2, S2 = _gpu(xq, 0.5, wq, 0.25, G, want_y=False)
    assert np.array_equal(q, q2) and np.array_equal(S.view(np.uint32), S2.view(np.uint32))


def test_zero_rows_and_columns_give_zero_groups():
    M, N, K, G = 128, 256, 128, 32
    xq = synth.fp8_operand_codes_np(M, K, 7)
    wq = synth.fp8_operand_codes_np(N, K, 8)
    xq[3] = 0x00                  # a zero row of X: every group of output row 3 is zero
    xq[4] = 0x80                  # negative zeros
    wq[32:64] = 0x00              # a zero group of columns in every row
    y, q, S = _gpu(xq, 1.0, wq, 1.0, G)
    assert (S[3] == 0).all() and (S[4] == 0).all() and (S[:, 1] == 0).all()
    assert (q[3] == 0).all() and (q[4] == 0).all() and (q[:, 32:64] == 0).all()
    _check(xq, 1.0, wq, 1.0, G, y, q, S)


@pytest.mark.parametrize("sx,sw", [(2.0 ** -70, 2.0 ** -63), (2.0 ** 40, 2.0 ** 41), (1e-3, 7.0)])
def test_extreme_scales(sx, sw):
    """Scales that put y near the bottom of the float32 range (subnormal
    group scales) or far up it; the quantization of the kernel's y stays exact."""
    M, N, K, G = 128, 128, 64, 16
    xq = synth.fp8_operand_codes_np(M, K, 9)
    wq = synth.fp8_operand_codes_np(N, K, 10)
    y, q, S = _gpu(xq, sx, wq, sw, G)
    assert np.isfinite(y).all()
    qk, Sk = oracle.absmax_quantize(y, G)
    assert np.array_equal(S.ravel().view(np.uint32), Sk.view(np.uint32))
    assert np.array_equal(q.ravel(), qk)
    if sx * sw > 2.0 ** -100:      # y normal: the summation bound holds as stated
        _check(xq, sx, wq, sw, G, y, q, S)


def test_every_code_pair():
    """Each of the 254 finite codes against each other one, through the tensor
    cores: K = 256 holds all codes (the two NaN codes replaced by zeros) and
    the rows of W are its cyclic shifts."""
    codes = np.arange(256, dtype=np.uint8)
    codes[[0x7F, 0xFF]] = 0
    M, N, K, G = 256, 256, 256, 64
    xq = np.stack([np.roll(codes, r) for r in range(M)])
    wq = np.stack([np.roll(codes[::-1], 3 * r) for r in range(N)])
    y, q, S = _gpu(xq, 1.0, wq, 1.0, G)
    _check(xq, 1.0, wq, 1.0, G, y, q, S)


@pytest.mark.parametrize("shape", [(8192, 4096, 4096), (4096, 11008, 4096), (4096, 4096, 11008)])
def test_llama7b_layer_shapes_on_sampled_rows(shape):
    """Llama-2-7B linear layers over 8192 / 4096 tokens (q/k/v/o projection,
    MLP up and down), G = 16 as for activations; rows sampled for the oracle."""
    M, N, K = shape
    G = 16
    xq = synth.fp8_operand_codes_np(M, K, 21)
    wq = synth.fp8_operand_codes_np(N, K, 22)
    y, q, S = _gpu(xq, 0.02, wq, 0.003, G)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(3).choice(M, 14, replace=False)]))
    _check(xq, 0.02, wq, 0.003, G, y[rows], q[rows], S[rows], rows=rows)
