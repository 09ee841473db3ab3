"""The oracle: a slow, plain fp64 CPU implementation of the PTPC-FP8 MoE layer.

TEST INFRASTRUCTURE ONLY. It is what the CUDA path is checked against and it
shares no code with that path. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it.
"""

from .fp8 import (E4M3_MAX, bf16_bits, bf16_from_bits, bf16_round,  # noqa: F401
                  e4m3_decode, e4m3_encode)
from .moe_ref import *  # noqa: F401,F403
from .norm_ref import add_rmsnorm_quant_ref, add_rmsnorm_ref, rsqrt_f32_rn  # noqa: F401
from .blockscale_ref import (BLOCK_K, BLOCK_N, SUBCHANNEL_K,  # noqa: F401
                             blockscale_matmul_ref, grouped_blockscale_ref,
                             quant_blocks_ref, quant_weight_blocks_ref,
                             subchannel_matmul_ref)
