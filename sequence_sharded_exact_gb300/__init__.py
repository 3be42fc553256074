"""GB300-native Ring Attention: blockwise exact attention over n virtual sequence shards.

The compute path is the C-ABI library ``libringattn.so`` (hand-written sm_103a CUDA kernels); this
package is a thin binding over it.  Importing the package does not load the library; the first
call does, and fails loudly if the library has not been built (``python -c "import
__graft_entry__ as g; g.build()"``).
"""
from .binding import (  # noqa: F401
    RingAttnError,
    bwd_workspace_size,
    device_check,
    device_status,
    fwd,
    fwd_f32out,
    fwd_host,
    fwd_stepwise,
    fwd_tile_visits,
    bwd,
    bwd_f32out,
    bwd_tile_visits,
    bwd_static_scratch,
    bwd_static_scratch_capacity,
    fwd_path,
    bwd_path,
    bwd_preprocess,
    block_bwd,
    block_fwd,
    block_rope,
    f32_add,
    f32_convert,
    f32_zero,
    library,
    lse_merge,
    ring_step_fwd,
    ring_step_fwd_accumulate,
    rope,
    selftest_bounded_wait,
    shard_tiles,
    ulysses_a2a,
    ulysses_bwd,
    ulysses_fwd,
)
from .autograd import ring_attention  # noqa: F401
from .ring import RingAttention, ring_attention_distributed  # noqa: F401
