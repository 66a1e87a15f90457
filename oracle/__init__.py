"""CPU oracles of the routed-expert block-quantized MoE FFN: numpy (float64) and C++.

TEST INFRASTRUCTURE. Only the test suite, `__graft_entry__.smoke()` and the
benchmark's `cpu_baseline` / `--impl reference` legs may import or call anything
here. It shares no code, tables or helpers with the CUDA library under
`block_quantized_moe_gb300/`, and neither imports the other.

Parity status per function (what pins it is in tests/test_oracle_*.py):
  formats.encode_e4m3 / decode_e4m3   pinned: OCP table values, torch float8_e4m3fn (exhaustive)
  formats.encode_e2m1 / decode_e2m1   pinned: OCP E2M1 magnitudes, every midpoint, saturation
  formats.round_to_bf16               pinned: torch bfloat16 conversion
  moe.quantize_act_fp8 / weight_fp8   pinned: closed forms (a 448 code in every nonzero group,
                                      exact power-of-two scales, round trip of representable values)
  moe.quantize_nvfp4                  pinned: closed forms (exact block/global scales, 6.0 codes)
  moe.quantize_mxfp8 / mx_shared_exp  pinned: closed forms (shared exponents, exact blocks, the
                                      clamp to 448, zero and partial blocks), floor(log2) from the
                                      fp32 bit pattern, torch float8_e4m3fn on the scaled values,
                                      the error bound, a brute-force MXFP8 FFN per element
  moe.segment_routes                  pinned: brute-force double loop, invariants
  moe.gather_rows_scales              pinned: identity map, duplicate rows, empty map
  moe.gemm_rows / moe_forward         pinned: brute-force dense FFN per token, one-hot columns,
                                      inactive-slot invariants
  moe.silu_mul                        pinned: scipy.special.expit, closed-form points
  moe.combine                         pinned: single route of weight 1, all inactive
  moe.pick_tile                       pinned: the dsfp4 page's table (tests/golden)
  slots.step                          pinned: a worked example, closed-form cases (empty pool,
                                      no fetch budget, slots used this step), invariants on
                                      random step sequences against the minimum-(usage, slot)
                                      formulation of the victim choice
  cpu (cpu_oracle.cpp)                the same definitions written again in plain C++17 with
                                      std::thread; pinned to the numpy oracle above (codes,
                                      scales, indices and bytes bit for bit; FFN outputs to
                                      float64 rounding) and to the same closed forms
"""
from . import formats, moe, slots  # noqa: F401
