"""GB300-native causal FP8 / BF16 prefill attention with the ZYFA numerics (Lean P, per-64-key
power-of-two block scaling, rounded-row-sum normalisation).

The compute path is the C-ABI library ``libzyfa.so`` built from ``csrc/`` for sm_103a; this package
only marshals arguments to it.  Importing the package does not load the library: the first call
does, and it raises if the library is missing.
"""
from .api import (ZyfaError, flash_attn_func, hadamard_quantize_e4m3, hadamard_quantize_qk_e4m3,  # noqa: F401
                  library_path, load_library, zyfa_attn_fwd_causal, zyfa_attn_fwd_causal_ex, zyfa_check_errors,
                  zyfa_kernel_launches)
