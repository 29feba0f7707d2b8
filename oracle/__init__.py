"""CPU oracle (test infrastructure): plain float64 numpy definitions of the sharded projection.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The CUDA product path never does.
"""
from .tp_oracle import *  # noqa: F401,F403
from .tp_oracle import (COLWISE, ROWWISE, PlanRejected, attention_core, bf16_to_f64,  # noqa: F401
                        check_plan, colwise_forward, combine_gather, combine_reduce, f64_to_bf16,
                        gelu_tanh, linear, mlp_forward, packed_block_sizes, rowwise_forward,
                        rowwise_partials, rowwise_split_input_forward, shard, shard_shape, silu, swiglu,
                        transformer_block_forward, single_stream_block_forward,
                        attention_block_forward, split_qkv, apply_act)
