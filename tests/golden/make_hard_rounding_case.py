"""Write hard_rounding_case.txt: the stored state of one element whose
dequantized moment is a hard fp32 rounding at a cancellation-driven group
minimum.

It replays the float64 oracle along the seeded 4096 x 4096 trajectory (the
input generator of coat_fp8_adamw_gb300.synth; about 80 s of CPU) to the
state before step 50 and records the element that is the smallest |m_t| of
group 8306 at that step.  Only the oracle and the input generator run here.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "..", ".."))
import oracle  # noqa: E402
from coat_fp8_adamw_gb300 import synth  # noqa: E402

STEP, GROUP = 50, 8306


def main():
    wl = synth.workload("mat4096")
    G, hp = wl.G, synth.HYPER
    w = synth.init_weights_np(wl)
    mq, vq, meta = synth.zero_state_np(wl.n, G)
    for t in range(1, STEP):
        oracle.adamw_step(w, synth.grad_np(wl, t), mq, vq, meta, G, hp["beta1"], hp["beta2"],
                          hp["lr"], hp["eps"], hp["weight_decay"], t)
    g = synth.bf16_bits_to_f32(synth.grad_np(wl, STEP))
    sl = slice(GROUP * G, GROUP * G + G)
    prev = oracle.dre_dequantize(mq[sl], meta[GROUP:GROUP + 1, 0], meta[GROUP:GROUP + 1, 1], G)
    b1 = float(np.float32(hp["beta1"]))
    m = (b1 * prev.astype(np.float64) + (1.0 - b1) * g[sl].astype(np.float64)).astype(np.float32)
    a = np.abs(m)
    j = int(np.argmin(np.where(a > 0, a, np.inf)))
    S, k = np.float32(meta[GROUP, 0]), np.float32(meta[GROUP, 1])
    lines = [
        "# One hard fp32 rounding of a dequantized first moment, written by",
        "# make_hard_rounding_case.py from the float64 oracle's 4096 x 4096 trajectory",
        f"# (state before step {STEP}, group {GROUP}, the element holding the group's",
        "# smallest |m_t|).  The value sign(q) (|E4M3(q)| S)^(1/k) lies within 3e-7",
        "# ulp of an fp32 rounding midpoint (COAT review page, section 3: the",
        "# dequantized tensor is X_FP32), and m_t = beta1 prev + (1 - beta1) g cancels",
        "# it about 23-fold.",
        "# code S_bits k_bits prev_bits g_bits",
        f"{int(mq[GROUP * G + j])} {int(S.view(np.uint32))} {int(k.view(np.uint32))} "
        f"{int(np.float32(prev[j]).view(np.uint32))} {int(np.float32(g[GROUP * G + j]).view(np.uint32))}",
    ]
    with open(os.path.join(HERE, "hard_rounding_case.txt"), "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
