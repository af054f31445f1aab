"""GPU parity of the fused FP8 AdamW + DRE step against the float64 oracle.

Every GPU call goes through the C ABI (ctypes binding).  Inputs come from the
seeded generators in coat_fp8_adamw_gb300.synth or from the oracle's own
trajectory: the GPU never produces an input of the oracle.  Multi-step runs
are teacher-forced the other way round: at step t the GPU starts from the
oracle's state after step t-1 and its output is compared with the oracle's
state after step t.
"""
import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

pytestmark = pytest.mark.gpu
HP = synth.HYPER


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.view(dtype)


def gpu_step(w, g_bits, mq, vq, meta, G, step, hp=HP):
    w_d = _dev(w.copy())
    g_d = _dev(g_bits.view(np.int16), torch.bfloat16)
    mq_d, vq_d, meta_d = _dev(mq.copy()), _dev(vq.copy()), _dev(meta.copy())
    coat.coat_fp8_adamw_step(w_d, g_d, mq_d, vq_d, meta_d, G, hp["beta1"], hp["beta2"], hp["lr"],
                             hp["eps"], hp["weight_decay"], step)
    torch.cuda.synchronize()
    return w_d.cpu().numpy(), mq_d.cpu().numpy(), vq_d.cpu().numpy(), meta_d.cpu().numpy()


def oracle_step(w, g_bits, mq, vq, meta, G, step, hp=HP):
    w, mq, vq, meta = w.copy(), mq.copy(), vq.copy(), meta.copy()
    oracle.adamw_step(w, g_bits, mq, vq, meta, G, hp["beta1"], hp["beta2"], hp["lr"], hp["eps"],
                      hp["weight_decay"], step)
    return w, mq, vq, meta


def check(gpu, ref, label):
    stats = {}
    stats.update(P.compare_w(gpu[0], ref[0], f"{label} w"))
    stats["m"] = P.compare_codes(gpu[1], ref[1], f"{label} m codes")
    stats["v"] = P.compare_codes(gpu[2], ref[2], f"{label} v codes")
    stats["meta_m"] = P.compare_meta(gpu[3][:, 0], gpu[3][:, 1], ref[3][:, 0], ref[3][:, 1],
                                     f"{label} (S_m, k_m)")
    stats["meta_v"] = P.compare_meta(gpu[3][:, 2], gpu[3][:, 3], ref[3][:, 2], ref[3][:, 3],
                                     f"{label} (S_v, k_v)")
    print(label, stats)
    return stats


def test_tiny_trajectory_teacher_forced():
    wl = synth.workload("tiny")
    w = synth.init_weights_np(wl)
    mq, vq, meta = synth.zero_state_np(wl.n, wl.G)
    for t in range(1, 11):
        g = synth.grad_np(wl, t)
        ref = oracle_step(w, g, mq, vq, meta, wl.G, t)
        gpu = gpu_step(w, g, mq, vq, meta, wl.G, t)
        check(gpu, ref, f"tiny t={t}")
        # edge groups of this workload: group 30 all-zero, group 31 one non-zero
        assert not gpu[1][30 * 128:31 * 128].any() and gpu[3][30, 0] == 0 and gpu[3][30, 1] == 1
        nz = np.nonzero(gpu[1][31 * 128:32 * 128])[0]
        assert gpu[3][31, 1] == 1.0 and np.all(gpu[1][31 * 128 + nz] & 0x7F == 0x7E)
        w, mq, vq, meta = ref


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_adamw_like_state_every_group_size(G):
    n = 4096 * 3 + 77                       # several CTAs and a ragged tail
    rng = np.random.default_rng(G)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2, n)).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, 100 + G, oracle)
    ref = oracle_step(w, g, mq, vq, meta, G, 7)
    gpu = gpu_step(w, g, mq, vq, meta, G, 7)
    check(gpu, ref, f"random G={G}")


@pytest.mark.parametrize("G", [16, 64, 128, 256])
def test_many_tiles_per_cta_with_ragged_tail(G):
    """Enough parameters that every persistent CTA of the step kernel runs
    several tiles of its double-buffered pipeline (more than 2048 parameters
    times three CTAs per SM times the SM count), with a ragged last tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 2048 * 3 * sms * 3 + 2048 * 5 + 333
    rng = np.random.default_rng(1000 + G)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2, n)).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, 200 + G, oracle)
    check(gpu_step(w, g, mq, vq, meta, G, 9), oracle_step(w, g, mq, vq, meta, G, 9), f"tiles G={G}")


@pytest.mark.parametrize("n", [1, 5, 16, 17, 127, 128, 129, 255, 4097])
def test_small_and_ragged_sizes(n):
    G = 128
    rng = np.random.default_rng(n)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, n, oracle)
    check(gpu_step(w, g, mq, vq, meta, G, 2), oracle_step(w, g, mq, vq, meta, G, 2), f"n={n}")


def test_mat4096_teacher_forced():
    wl = synth.workload("mat4096")
    w = synth.init_weights_np(wl)
    mq, vq, meta = synth.zero_state_np(wl.n, wl.G)
    for t in range(1, 4):
        g = synth.grad_np(wl, t)
        ref = oracle_step(w, g, mq, vq, meta, wl.G, t)
        gpu = gpu_step(w, g, mq, vq, meta, wl.G, t)
        check(gpu, ref, f"mat4096 t={t}")
        w, mq, vq, meta = ref


def _edge_inputs(G=128):
    """Groups whose moments hit every special case of the per-group parameters."""
    groups = []
    rng = np.random.default_rng(3)
    z = np.zeros(G, np.float32)
    groups.append(z.copy())                                   # all-zero gradient
    one = z.copy(); one[17] = 3e-3; groups.append(one)        # single non-zero
    eq = np.full(G, 2e-3, np.float32); eq[::2] *= -1; groups.append(eq)   # equal magnitudes
    near = (1e-3 * (1 + 0.05 * rng.random(G))).astype(np.float32); groups.append(near)  # R_X ~ 1.05: cap
    sub = np.full(G, 1e-39, np.float32); sub[::3] = 3e-39; groups.append(sub)           # fp32 subnormal g
    tiny = (rng.standard_normal(G) * 1e-30).astype(np.float32); groups.append(tiny)     # S guard
    big = (rng.standard_normal(G) * 30.0).astype(np.float32); groups.append(big)        # large values
    wide = (np.exp(rng.uniform(-20, 0, G)) * np.sign(rng.standard_normal(G))).astype(np.float32)
    groups.append(wide)                                       # R_X > R_E4M3: k < 1
    half = (rng.standard_normal(G) * 1e-3).astype(np.float32); half[G // 2:] = 0; groups.append(half)
    return np.concatenate(groups)


def test_edge_groups_zero_state_and_warm():
    G = 128
    gf = _edge_inputs(G)
    n = gf.size
    g = synth.f32_to_bf16_bits(gf)
    w = np.linspace(-0.05, 0.05, n).astype(np.float32)
    mq, vq, meta = synth.zero_state_np(n, G)
    for t in range(1, 4):
        ref = oracle_step(w, g, mq, vq, meta, G, t)
        gpu = gpu_step(w, g, mq, vq, meta, G, t)
        check(gpu, ref, f"edge t={t}")
        w, mq, vq, meta = ref
    # all-zero group stays at the initial record; single non-zero group has k = 1
    assert gpu[3][0, 0] == 0 and gpu[3][0, 1] == 1 and gpu[3][1, 1] == 1 and gpu[3][1, 3] == 1


def test_large_step_count_and_hyperparameters():
    n, G = 4096 + 33, 64
    rng = np.random.default_rng(11)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, 9, oracle)
    for hp, step in ((dict(HP), 1_000_000), (dict(beta1=0.5, beta2=0.999, lr=3e-3, eps=1e-6,
                                                   weight_decay=0.0), 3)):
        check(gpu_step(w, g, mq, vq, meta, G, step, hp), oracle_step(w, g, mq, vq, meta, G, step, hp),
              f"hp={hp} t={step}")


def test_in_place_and_stream_semantics():
    """The step runs on the caller's stream, in place, and is deterministic."""
    n, G = 8192 + 5, 128
    rng = np.random.default_rng(12)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, 12, oracle)
    a = gpu_step(w, g, mq, vq, meta, G, 4)
    s = torch.cuda.Stream()
    w_d, g_d = _dev(w.copy()), _dev(g.view(np.int16), torch.bfloat16)
    mq_d, vq_d, meta_d = _dev(mq.copy()), _dev(vq.copy()), _dev(meta.copy())
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        coat.coat_fp8_adamw_step(w_d, g_d, mq_d, vq_d, meta_d, G, HP["beta1"], HP["beta2"],
                                 HP["lr"], HP["eps"], HP["weight_decay"], 4, stream=s)
    s.synchronize()
    for x, y in zip(a, (w_d.cpu().numpy(), mq_d.cpu().numpy(), vq_d.cpu().numpy(), meta_d.cpu().numpy())):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_argument_errors_on_device():
    n, G = 256, 128
    w = torch.zeros(n, device="cuda")
    g = torch.zeros(n, device="cuda", dtype=torch.bfloat16)
    mq = torch.zeros(n, device="cuda", dtype=torch.uint8)
    vq = torch.zeros(n, device="cuda", dtype=torch.uint8)
    meta = torch.zeros(2, 4, device="cuda")
    L = coat.lib()
    # a group size that is not a power of two is refused by the library itself
    st = L.coat_fp8_adamw_step(w.data_ptr(), g.data_ptr(), mq.data_ptr(), vq.data_ptr(),
                               meta.data_ptr(), n, 96, 0.9, 0.95, 1e-4, 1e-8, 0.1, 1, None)
    assert st == 3
    with pytest.raises(ValueError):   # the binding checks the record count first
        coat.coat_fp8_adamw_step(w, g, mq, vq, meta, 96, 0.9, 0.95, 1e-4, 1e-8, 0.1, 1)
    with pytest.raises(coat.CoatError) as e:
        coat.coat_fp8_adamw_step(w, g, mq, vq, meta, G, 0.9, 0.95, 1e-4, 1e-8, 0.1, 0)
    assert e.value.status == 1
    # host memory is refused even though the call would otherwise be valid
    wh = torch.zeros(n)
    st = L.coat_fp8_adamw_step(wh.data_ptr(), g.data_ptr(), mq.data_ptr(), vq.data_ptr(),
                               meta.data_ptr(), n, G, 0.9, 0.95, 1e-4, 1e-8, 0.1, 1, None)
    assert st == 5
    # misaligned pointer
    wbig = torch.zeros(n + 4, device="cuda")
    st = L.coat_fp8_adamw_step(wbig.data_ptr() + 4, g.data_ptr(), mq.data_ptr(), vq.data_ptr(),
                               meta.data_ptr(), n, G, 0.9, 0.95, 1e-4, 1e-8, 0.1, 1, None)
    assert st == 2
    torch.cuda.synchronize()
