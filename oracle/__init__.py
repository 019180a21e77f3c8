"""CPU oracle for causal FP8 / BF16 prefill attention with the ZYFA numerics.

TEST INFRASTRUCTURE ONLY: this package is imported by ``tests/``, by ``__graft_entry__.smoke()`` and by
the CPU-baseline leg of ``bench.py``, and by nothing else.  It shares no code with the CUDA library and
never reads a value produced by it.

Functions and the passages they follow (page title, section):

* ``formats.e4m3_decode`` / ``e4m3_encode_rne_satfinite`` / ``bf16_round``: the OCP FP8 e4m3 and bfloat16
  encodings; the "+8 per doubling" property of e4m3 codes is the one the Lean-P bullet of
  "Три приёма" (spbcomputers.ru ZYFA article) relies on.
* ``exact_causal_attention`` (O1): causal softmax attention, float64 (ZYFA abstract, first sentences).
* ``leanp_causal_attention`` (O2): Lean P, per-64-key power-of-two scaling, rounded-row-sum
  normalisation (ZYFA abstract, techniques (1) and (3); "Три приёма"; "Tiga Trik").
* ``exactp_causal_attention`` (O2x): O2 with exact exponentiation and e4m3 rounding in place of Lean P,
  the baseline the pages compare Lean P with ("Tiga Trik": 5.9% vs 7.5% per probability).
* ``exactp_noblock_causal_attention`` (O2xn): O2x without the per-block scaling, every probability
  rounded against the row's running reference exponent: the ablation of the per-64-key scaling
  ("Три приёма"; "Tiga Trik"), with the running reference a reading.
* ``return_lse=True`` on O1, O2, O2x, O2xn, O4: ln sum_j exp(s_ij) per row (flash_attn_func's softmax_lse).
* ``plain_fp8_causal_attention`` (O3): exact-exponential FP8 softmax, comparison only.
* ``bf16_causal_attention`` (O4): the BF16 twin (the pages give no BF16 numerics; plainest reading).
* ``hadamard``: Hadamard rotation of Q and K before quantisation (spbcomputers.ru ZYFA article, FAQ
  "Что даёт поворот Адамара?"; captivela ZYFA article, "Angka Nyata").
"""
from .formats import (E4M3_MAX, bf16_bits_to_float, bf16_round, e4m3_decode,  # noqa: F401
                      e4m3_encode_rne_satfinite, fl32)
from .attention import (LEANP_C0, SCALE_BLOCK, bf16_causal_attention,  # noqa: F401
                        bf16_round_f64, bf16_score_scale, default_softmax_scale, dequant_e4m3,
                        exact_causal_attention, exactp_causal_attention, exactp_code,
                        exactp_noblock_causal_attention, exactp_noblock_weights, fp8_score_scale,
                        leanp_causal_attention, leanp_code,
                        leanp_row_weights, plain_fp8_causal_attention, rel_l2)
from .hadamard import (fwht_f32, hadamard_block, hadamard_matrix, hadamard_quantize_e4m3,  # noqa: F401
                       rotate)
