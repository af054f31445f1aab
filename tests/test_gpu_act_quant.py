"""Per-group (1 x G) FP8 activation quantization with the transposed second
output, on the GPU through the C ABI, against the oracle."""
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


def _activation(M, N, seed):
    """bf16 activations with a per-row scale spread and a few large outliers."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, N)) * 10.0 ** rng.uniform(-3, 1, (M, 1))
    x[rng.random((M, N)) < 1e-3] *= 100.0
    x[0, :] = 0.0                                   # an all-zero row: all-zero groups
    return synth.f32_to_bf16_bits(x.astype(np.float32)).reshape(M, N)


def _gpu(bits, G, transposed=True):
    M, N = bits.shape
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    qt = torch.empty((N, M), dtype=torch.uint8, device="cuda") if transposed else None
    S = torch.empty((M, N // G), dtype=torch.float32, device="cuda")
    coat.coat_act_quantize_fp8(x, G, q, S, qt)
    torch.cuda.synchronize()
    return q.cpu().numpy(), (qt.cpu().numpy() if transposed else None), S.cpu().numpy()


@pytest.mark.parametrize("G", [4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("shape", [(208, 384), (64, 128), (16, 256), (80, 640)])
def test_matches_oracle(G, shape):
    M, N = shape
    bits = _activation(M, N, G + M)
    q, qt, S = _gpu(bits, G)
    qo, qto, So = oracle.act_quantize(bits, G)
    assert np.array_equal(S, So), "scales must be bit-identical"
    P.assert_codes_equal(q, qo, f"q G={G} {shape}")
    assert np.array_equal(qt, q.T), "the second output is the first one transposed"


def test_ragged_column_tile_and_no_transpose():
    G, M, N = 16, 48, 400            # 400 = 3 tiles of 128 + 16 columns
    bits = _activation(M, N, 9)
    q, _, S = _gpu(bits, G, transposed=False)
    qo, _, So = oracle.act_quantize(bits, G)
    assert np.array_equal(S, So)
    P.assert_codes_equal(q, qo, "ragged q")
    q2, qt2, _ = _gpu(bits, G)
    assert np.array_equal(q2, q) and np.array_equal(qt2, q.T)


def test_large_tensor_sampled_rows():
    G, M, N = 16, 16384, 4096        # a 64M-element activation, checked on sampled rows
    rng = np.random.default_rng(2)
    x = torch.randn(M, N, generator=torch.Generator(device="cuda").manual_seed(3), device="cuda")
    x = (x * torch.pow(10.0, torch.rand(M, 1, device="cuda") * 4 - 3)).to(torch.bfloat16)
    q = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    qt = torch.empty((N, M), dtype=torch.uint8, device="cuda")
    S = torch.empty((M, N // G), dtype=torch.float32, device="cuda")
    coat.coat_act_quantize_fp8(x, G, q, S, qt)
    rows = np.sort(rng.choice(M, 64, replace=False))
    bits = x[rows].view(torch.int16).cpu().numpy().view(np.uint16)
    qo, _, So = oracle.act_quantize(bits, G)
    assert np.array_equal(S[rows].cpu().numpy(), So)
    P.assert_codes_equal(q[rows].cpu().numpy(), qo, "sampled rows")
    cols = np.sort(rng.choice(N, 64, replace=False))
    assert torch.equal(qt[cols], q[:, cols].T)


def test_argument_errors():
    x = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
    S = torch.empty(64 * 128 // 16, dtype=torch.float32, device="cuda")
    L = coat.lib()
    assert L.coat_act_quantize_fp8(x.data_ptr(), 64, 128, 2, q.data_ptr(), None, S.data_ptr(), None) == 3
    assert L.coat_act_quantize_fp8(x.data_ptr(), 60, 128, 16, q.data_ptr(), None, S.data_ptr(), None) == 1
    assert L.coat_act_quantize_fp8(x.data_ptr(), 64, 120, 16, q.data_ptr(), None, S.data_ptr(), None) == 1
    assert L.coat_act_quantize_fp8(x.data_ptr(), 64, 128, 16, q.data_ptr(), None, S.data_ptr(), None) == 0


def _midpoint_groups():
    """Groups [max, x, 0, 0] of bf16 values with 448 x / max exactly an E4M3
    midpoint; S = max / 448 is rarely exact, so the exact quotient x / S lies
    just beside the midpoint while its float32 rounding is often the midpoint."""
    dec = np.array([oracle.e4m3_decode(c) for c in range(128)])
    mids = sorted(set(((dec[1:127] + dec[0:126]) / 2).tolist()))
    groups = []
    for c in range(3, 256, 2):
        for a in (-3, 0, 2):
            mx = c * 2.0 ** a
            for m in mids:
                x = m * mx / 448
                b = synth.f32_to_bf16_bits(np.array([x], np.float32))
                if float((b.astype(np.uint32) << 16).view(np.float32)[0]) == x:
                    groups.append([mx, x, 0.0, 0.0])
    return np.array(groups, np.float32)


@pytest.mark.parametrize("scale", [1.0, -(2.0 ** -112)])
def test_quotients_beside_a_midpoint_round_like_the_exact_quotient(scale):
    """Both quantizers must round the exact quotient, not its float32 rounding;
    also for negative values around 2^-120, where the activation quantizer
    scales the midpoint test into range."""
    G = 4
    grp = _midpoint_groups() * np.float32(scale)
    back = (synth.f32_to_bf16_bits(grp).astype(np.uint32) << 16).view(np.float32).reshape(grp.shape)
    grp = grp[np.all(back == grp, axis=1)]              # every value still exact in bf16
    grp = grp[: (len(grp) // 64) * 64]                  # rows of 16 elements, M a multiple of 16
    x = grp.reshape(-1, 16)
    S32 = (np.abs(x[:, ::4]).astype(np.float64) / 448).astype(np.float32)
    naive = torch.from_numpy((x[:, 1::4] / S32).astype(np.float32)).to(torch.float8_e4m3fn)
    qo, _, So = oracle.act_quantize(synth.f32_to_bf16_bits(x).reshape(x.shape), G)
    disagree = (naive.view(torch.uint8).numpy() != qo[:, 1::4]).sum()
    assert disagree > 100, "the inputs must include quotients whose float32 rounding misleads"
    q, _, S = _gpu(synth.f32_to_bf16_bits(x).reshape(x.shape), G)
    assert np.array_equal(S, So)
    assert np.array_equal(q, qo), f"{int((q != qo).sum())} codes differ from the oracle's"
    xd = torch.from_numpy(x.ravel().copy()).cuda()
    qa = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    Sa = torch.empty(x.size // G, dtype=torch.float32, device="cuda")
    coat.coat_fp8_quantize_absmax(xd, G, qa, Sa)
    qao, _ = oracle.absmax_quantize(x.ravel(), G)
    assert np.array_equal(qa.cpu().numpy(), qao)
