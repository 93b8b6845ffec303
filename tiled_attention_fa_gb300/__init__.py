"""GB300-native (sm_103a) tiled online-softmax attention, forward and backward.

The compute path is the C-ABI library ``libfa_gb300.so`` (hand-written CUDA:
TMA, tcgen05 MMA with TMEM accumulators, warp-specialised pipelines); this
package only marshals torch tensors into it.  Build the library with
``python -m tiled_attention_fa_gb300.build``.
"""

from .api import (  # noqa: F401
    DecodeHostRunner,
    Fp8HostRunner,
    HostPipeline,
    HostRunner,
    alloc_workspace,
    attention_backward,
    bwd,
    bwd_main,
    bwd_postprocess,
    bwd_preprocess,
    check_device_error,
    alloc_decode_workspace,
    decode,
    decode_merge,
    decode_slices,
    decode_workspace_size,
    fwd,
    fwd_fp8,
    workspace_size,
)

__all__ = ["fwd", "bwd_preprocess", "bwd", "attention_backward", "bwd_main", "bwd_postprocess", "workspace_size",
           "alloc_workspace", "check_device_error", "HostRunner", "HostPipeline", "decode", "decode_workspace_size",
           "decode_slices", "decode_merge", "alloc_decode_workspace", "DecodeHostRunner", "fwd_fp8", "Fp8HostRunner"]
