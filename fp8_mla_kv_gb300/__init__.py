"""libmlasparse: FP8 MLA KV cache writer and sparse top-k MLA decode for GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind a C ABI
(``include/mlasparse.h``); ``fp8_mla_kv_gb300.mlasparse`` is the thin Python
binding with the same function names. The shared library is loaded on first
use, and every call fails loudly if it is missing: there is no CPU fallback.
"""

ROW_BYTES = 656
ROW_BYTES_NOPE = 528
LATENT_DIM = 512
ROPE_DIM = 64
