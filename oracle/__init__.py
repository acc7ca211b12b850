"""CPU oracle for block-wise masked-diffusion decoding (test infrastructure).

This package is the plain, slow, obviously correct statement of what one
denoising step computes.  It exists to check the CUDA path and to time a
CPU baseline; nothing in the product imports it.  Only the tests, the
smoke check and the benchmark's CPU-baseline leg may call it.

Arithmetic is fp32 (NumPy; its matmul is the one library primitive used),
over bf16-rounded weights and context K/V.  See `oracle.decode` for each
function and the passage it follows.

Parity status of each function:

* attention, confidence/argmax, commit, RMSNorm, SwiGLU, full step:
  pinned by the tests under tests/ (double-precision brute force on tiny
  shapes, closed forms, invariants, exhaustive commit enumeration).
* near-tie flags (which positions the parity tests may waive): pinned by
  hand-derived cases in tests/golden/near_tie_cases.txt and by a soundness
  property (perturbing logits and confidences within half the thresholds
  changes the commit only at flagged positions).
* The denoiser's weights are synthetic: end-to-end token ids have no
  published value to match, so beyond the pins above they are checked
  only for agreement between this oracle and the CUDA path.
"""
from .decode import (  # noqa: F401
    TIE_CONF_GAP,
    TIE_GAMMA_GAP,
    TIE_LOGIT_GAP,
    MODE_MOCK_AR,
    MODE_STEPS,
    MODE_THRESHOLD,
    MODE_TOPK,
    OracleModel,
    append_block,
    StepResult,
    block_attention,
    commit,
    decode_block,
    denoise_step,
    linear,
    lm_head_select,
    near_tie_flags,
    near_tie_positions,
    top2_gap,
    tower_causal_attention,
    rmsnorm,
    rope,
    round_bf16,
    select_from_logits,
    steps_schedule_k,
    with_param,
    silu,
)
