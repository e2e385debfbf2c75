"""CPU oracle for the fused multi-tensor AdamW step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (``compact_state_gb300``)
never imports, calls or links it, and this package never imports the product.

The oracle is plain numpy in float64, written from the method page
"融合优化器与状态精度：把参数更新的读写和状态分开优化" (Fused Optimizers and State
Precision, xuujii.github.io ai-infra-kb M041):

* ``formats``    -- round-to-nearest-even into fp32 / bf16 / fp16 storage
                    (section 05 names 16-bit moments; rounding mode is IEEE RNE).
* ``int8_block`` -- the teaching signed block codec of section 05
                    (scale = max|x|/127, q = round(x/scale), x ~ q*scale,
                    all-zero blocks handled separately).
* ``dynamic8``   -- the non-linear 8-bit codebook variant of section 05 (the
                    published dynamic tree quantization; signed for m,
                    unsigned for v), one fp32 absmax per 256-element block.
                    ``int8_block`` also holds the unsigned linear variant for v.
* ``adamw``      -- the AdamW update of section 02 in the page's own order, the
                    three-separate-loops form of section 04, and the step/skip
                    contract of sections 02, 03 and 06 (grad=None skips a tensor,
                    an overflowing step leaves everything untouched).
* ``state_bytes``-- the optimizer-state byte ledger (section 05 payloads, and the
                    state-memory figures of the ApexW Unsloth benchmark page).

What pins each function (tests marked ``not gpu``):

* ``formats.round_to``      numpy's own float32/float16 casts and torch's CPU
                            bfloat16 cast (library routines), special values.
* ``int8_block``            the reconstruction bound |x - q*scale| <= scale/2,
                            max|x| -> +-127, zero blocks, exact multiples, and
                            brute-force nearest-code search on small blocks.
* ``adamw.adamw_update``    the page's worked example (tests/golden), the
                            constant-gradient closed form, and the unrolled-sum
                            closed form of the moments and of theta evaluated in
                            exact rational / high-precision decimal arithmetic.
* ``adamw.oracle_step``     None / zero-grad / overflow invariants, the
                            unscale-by-power-of-two identity, and equality with
                            the three-loop form.
* ``state_bytes``           the benchmark page's 185.501 / 92.751 / 47.101 MB.
* ``int8_block`` (unsigned) the bound, max -> 255, exact multiples, brute-force
                            nearest code, half the signed codec's error.
* ``dynamic8``              the table's structure from its bit layout (decade
                            tops against fp32(10^-E), equal in-decade steps),
                            brute-force nearest-code search, the per-decade
                            error bound, small values kept next to an outlier.
"""
from . import formats, int8_block, dynamic8, adamw, state_bytes  # noqa: F401
from .adamw import (TensorState, adamw_update, oracle_step,  # noqa: F401
                    oracle_step_three_loops, new_state)
