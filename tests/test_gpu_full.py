"""Full-size parity: one fused step over a whole model-shaped parameter set on
the GPU (the launch the benchmark times), checked on sampled groups.

The parameter sets are drawn on the device by the seeded generators.  Every
group starts from a random synthetic state; the sampled groups instead carry
a state the oracle produced itself by warming them from zero for several
steps with the same full-size gradients (groups are independent, so this is
exact).  The GPU then runs one step over the whole buffer, and the sampled
groups are compared with the oracle's step from the same inputs.
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


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,G,warm", [("olmo1b", 128, 20), ("llama7b", 128, 10),
                                         ("llama13b", 16, 4), ("llama13b", 32, 4),
                                         ("llama13b", 64, 4), ("llama13b", 128, 4),
                                         ("llama13b", 256, 4)])
def test_full_size_sampled(name, G, warm):
    dev = torch.device("cuda:0")
    wl = synth.workload(name, G)
    n = wl.n
    ng = coat.num_groups(n, G)
    w = synth.init_weights_torch(wl, dev)
    mq, vq, meta = synth.random_state_torch(n, G, seed=wl.seed, device=dev)
    groups = synth.sample_groups(ng, 2048 if G >= 64 else 8192, seed=wl.seed)
    idx = (groups[:, None] * G + np.arange(G)[None, :]).ravel()
    idx = idx[idx < n]
    idx_t = torch.from_numpy(idx).to(dev)
    grp_t = torch.from_numpy(groups).to(dev)

    # oracle-warmed state in the sampled groups
    ws = w[idx_t].cpu().numpy()
    mqs, vqs, metas = synth.zero_state_np(idx.size, G)
    for t in range(1, warm + 1):
        gs = _bits(synth.grad_torch(wl, t, dev)[idx_t])
        oracle.adamw_step(ws, gs, mqs, vqs, metas, G, HP["beta1"], HP["beta2"], HP["lr"],
                          HP["eps"], HP["weight_decay"], t)
    w[idx_t] = torch.from_numpy(ws).to(dev)
    mq[idx_t] = torch.from_numpy(mqs).to(dev)
    vq[idx_t] = torch.from_numpy(vqs).to(dev)
    meta[grp_t] = torch.from_numpy(metas).to(dev)

    t = warm + 1
    g = synth.grad_torch(wl, t, dev)
    gs = _bits(g[idx_t])
    torch.cuda.synchronize()
    coat.coat_fp8_adamw_step(w, g, mq, vq, meta, G, HP["beta1"], HP["beta2"], HP["lr"], HP["eps"],
                             HP["weight_decay"], t)
    torch.cuda.synchronize()
    out = (w[idx_t].cpu().numpy(), mq[idx_t].cpu().numpy(), vq[idx_t].cpu().numpy(),
           meta[grp_t].cpu().numpy())
    # the rest of the buffer was updated too (no NaN, codes finite)
    assert torch.isfinite(w).all().item()
    assert not ((mq & 0x7F) == 0x7F).any().item() and not ((vq & 0x7F) == 0x7F).any().item()
    assert torch.isfinite(meta).all().item() and (meta[:, 1] > 0).all().item()
    del w, g, mq, vq, meta
    torch.cuda.empty_cache()

    oracle.adamw_step(ws, gs, mqs, vqs, metas, G, HP["beta1"], HP["beta2"], HP["lr"], HP["eps"],
                      HP["weight_decay"], t)
    st = {}
    st.update(P.compare_w(out[0], ws, f"{name} w"))
    st["m"] = P.compare_codes(out[1], mqs, f"{name} m codes")
    st["v"] = P.compare_codes(out[2], vqs, f"{name} v codes")
    st["meta_m"] = P.compare_meta(out[3][:, 0], out[3][:, 1], metas[:, 0], metas[:, 1], f"{name} m")
    st["meta_v"] = P.compare_meta(out[3][:, 2], out[3][:, 3], metas[:, 2], metas[:, 3], f"{name} v")
    print(name, G, st)
