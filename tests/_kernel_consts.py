"""Constants of the step kernel's source that tests check against the
hardware or a model (read from the source, so that the two cannot drift)."""
import os
import re

STEP_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", "coat_fp8_adamw_gb300",
                        "csrc", "adamw_dre_step.cu")


def kernel_ex2_bound() -> float:
    """The relative error of the SFU exp2 that the fast path's bound assumes (kEx2Err)."""
    with open(STEP_SRC) as fh:
        m = re.search(r"constexpr float kEx2Err = ([0-9.eE+-]+)f;", fh.read())
    assert m, "kEx2Err not found in the step kernel source"
    return float(m.group(1))
