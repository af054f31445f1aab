"""Host-side check of coat_round.cuh, the certain-rounding test and the
float64 recomputations meant for the exact path's rare hard roundings (CPU
only; the header also compiles for the device)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc")


def test_round_certain_is_never_wrong(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "round_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC,
                    os.path.join(ROOT, "tests", "native", "round_check.cpp"), "-o", str(exe), "-lm"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    stats = {k: float(v) for k, v in (kv.split("=") for kv in out.split())}
    print(stats)
    assert stats["random_wrong"] == 0 and stats["near_certain_wrong"] == 0
    assert stats["random_uncertain_frac"] < 1e-4        # about 2 eps / ulp = 2^-15
    assert stats["near_uncertain_frac"] > 0.2           # the uncertain branch is exercised
    assert stats["dequant_diff"] == 0 and stats["k_diff"] == 0
    # the division-free form of the test used for k
    assert stats["q_wrong"] == 0 and stats["q_uncertain_frac"] > 0.2


def test_header_compiles_for_the_device(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "use_round.cu"
    src.write_text(
        '#include "coat_round.cuh"\n'
        "__global__ void k(const float* in, float* out, int* flag) {\n"
        "    bool c = false;\n"
        "    out[0] = coat::df::round_certain(coat::df::F2{in[0], in[1]}, 0x1p-40f, c);\n"
        "    flag[0] = c;\n"
        "    out[1] = coat::df::dequant_f64(in[2], in[3], in[4]);\n"
        "    out[2] = coat::df::k_f64(in[5], in[6], 229376.0, 8.0, -125.0, 126.0);\n"
        "}\n")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-I", CSRC,
                    "-c", str(src), "-o", str(tmp_path / "use_round.o")], check=True)


def test_float64_recomputations_match_the_oracle(tmp_path):
    """The recomputations reproduce the oracle's definitions: its dequantized
    moments, and its k with the cap and the S-range guard, for groups of two
    magnitudes (max, min) spread over the whole range."""
    import ctypes

    import numpy as np

    import oracle
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "f64.cpp"
    src.write_text('#include "coat_round.cuh"\n'
                   'extern "C" float dq(float m, float s, float k) { return coat::df::dequant_f64(m, s, k); }\n'
                   'extern "C" float kk(float mx, float mn) {\n'
                   '    return coat::df::k_f64(mx, mn, 229376.0, 8.0, -125.0, 126.0); }\n')
    lib = tmp_path / "libf64.so"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", "-I", CSRC,
                    str(src), "-o", str(lib)], check=True)
    L = ctypes.CDLL(str(lib))
    L.dq.argtypes = [ctypes.c_float] * 3
    L.dq.restype = ctypes.c_float
    L.kk.argtypes = [ctypes.c_float] * 2
    L.kk.restype = ctypes.c_float
    rng = np.random.default_rng(33)
    dec = oracle.e4m3_decode_all()
    codes = rng.choice(np.array([c for c in range(1, 127) if c != 0x7F], np.uint8), 3000)
    S = np.exp2(rng.uniform(-120.0, 0.0, codes.size)).astype(np.float32)
    k = rng.uniform(0.6, 8.0, codes.size).astype(np.float32)
    for c, s, kv in zip(codes, S, k):
        want = oracle.dre_dequantize(np.array([c], np.uint8), np.array([s]), np.array([kv]), 1)[0]
        assert np.float32(L.dq(float(dec[c]), float(s), float(kv))) == want
    # (max, min) pairs: ordinary, capped (ratio below 4.68), guard-active (tiny or huge max)
    lmx = rng.uniform(-140.0, 120.0, 3000)
    ratio = np.where(rng.random(3000) < 0.2, rng.uniform(0.0, 2.2, 3000), rng.uniform(2.2, 40.0, 3000))
    for a, r in zip(lmx, ratio):
        mx = np.float32(2.0 ** a)
        mn = np.float32(2.0 ** (a - r))
        if not (mn > 0 and np.isfinite(mx)):
            continue
        g = oracle.dre_group(np.array([mx, mn], np.float32))
        assert np.float32(L.kk(float(mx), float(mn))) == np.float32(g["k"]), (float(mx), float(mn))


def _near_midpoint_dequant_cases(rng, N):
    dec = oracle_mod().e4m3_decode_all()
    finite = np.array([c for c in range(1, 127) if c != 0x7F], dtype=np.uint8)
    codes = rng.choice(finite, N)
    S = np.exp2(rng.uniform(-110.0, 0.0, N)).astype(np.float32)
    k = rng.uniform(0.6, 8.0, N).astype(np.float32)
    x = (np.abs(dec[codes]) * S.astype(np.float64)) ** (1.0 / k.astype(np.float64))
    ok = (x > 2.0 ** -126) & (x < 2.0 ** 127)
    frac = x / np.spacing(x.astype(np.float32)).astype(np.float64)
    dist = np.abs(frac - np.floor(frac) - 0.5)
    return codes, S, k, ok, dist


def oracle_mod():
    import oracle
    return oracle


def test_exact_path_dequant_matches_the_oracle_at_hard_roundings(tmp_path):
    """The step kernel's exact dequantization (host build of the same code)
    equals the oracle's correctly rounded fp32 value bit for bit, for values
    within 1e-5 ulp of an fp32 midpoint (decided by the float64 path), between
    1e-5 and 1e-3 ulp, and at random; the float64 path stays rare at random."""
    import _exact_path
    oracle = oracle_mod()
    exe = _exact_path.build(tmp_path)
    rng = np.random.default_rng(41)
    codes, S, k, ok, dist = _near_midpoint_dequant_cases(rng, 3_000_000)
    hard = np.nonzero(ok & (dist < 1e-5))[0][:80]
    medium = np.nonzero(ok & (dist >= 1e-5) & (dist < 1e-3))[0][:300]
    rand = np.nonzero(ok)[0][:20000]
    assert hard.size >= 30
    for name, idx in (("hard", hard), ("medium", medium), ("random", rand)):
        got, slow = _exact_path.dequant(exe, codes[idx], S[idx], k[idx])
        want = np.array([oracle.dre_dequantize(codes[i:i + 1], S[i:i + 1], k[i:i + 1], 1)[0]
                         for i in idx], np.float32)
        bad = np.nonzero(got.view(np.uint32) != np.abs(want).view(np.uint32))[0]
        assert bad.size == 0, (name, [(int(codes[idx[j]]), float(S[idx[j]]), float(k[idx[j]]))
                                      for j in bad[:5]])
        print(name, idx.size, "float64 path", int(slow.sum()))
        if name == "hard":
            assert slow.mean() > 0.5            # the band of doubt covers these
        if name == "random":
            assert slow.mean() < 1e-3


def test_exact_path_k_matches_the_oracle_at_hard_roundings(tmp_path):
    """The step kernel's k (host build of the same code) equals the oracle's
    bit for bit for k within 1e-5 ulp of an fp32 midpoint, at random, and where
    the cap or the S-range guard decides."""
    import _exact_path
    oracle = oracle_mod()
    exe = _exact_path.build(tmp_path)
    rng = np.random.default_rng(42)
    N = 3_000_000
    mx = np.exp2(rng.uniform(-40.0, 10.0, N)).astype(np.float32)
    mn = (mx.astype(np.float64) * np.exp2(-rng.uniform(2.3, 40.0, N))).astype(np.float32)
    kk = np.log(229376.0) / np.log(mx.astype(np.float64) / mn.astype(np.float64))
    frac = kk / np.spacing(kk.astype(np.float32)).astype(np.float64)
    dist = np.abs(frac - np.floor(frac) - 0.5)
    free = kk < 7.9
    hard = np.nonzero(free & (dist < 1e-5))[0][:60]
    rand = np.arange(3000)
    # guard-active (tiny or huge max) and cap-active (ratio below 4.68) pairs
    lmx = rng.uniform(-140.0, 120.0, 3000)
    ratio = np.where(rng.random(3000) < 0.3, rng.uniform(0.0, 2.3, 3000), rng.uniform(2.3, 40.0, 3000))
    emx = np.exp2(lmx).astype(np.float32)
    emn = np.exp2(lmx - ratio).astype(np.float32)
    keep = (emn > 0) & np.isfinite(emx) & (emx > 0)
    assert hard.size >= 30
    cases = [("hard", mx[hard], mn[hard]), ("random", mx[rand], mn[rand]),
             ("edges", emx[keep], emn[keep])]
    for name, a, b in cases:
        got, slow = _exact_path.kexp(exe, a, b)
        want = np.array([oracle.dre_group(np.array([x, y], np.float32))["k"] for x, y in zip(a, b)],
                        np.float32)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (name, [(float(a[j]), float(b[j]), float(got[j]), float(want[j]))
                                      for j in bad[:5]])
        print(name, a.size, "float64 path", int(slow.sum()))
        if name == "hard":
            # k's band of doubt is about 2^-43 (2 + |log2 max| + |log2 min|) /
            # log2 R_X relative: a good part of values within 1e-5 ulp of a
            # midpoint (6e-13 relative at most) lies inside it
            assert slow.mean() > 0.25
        if name == "random":
            assert slow.mean() < 2e-3
