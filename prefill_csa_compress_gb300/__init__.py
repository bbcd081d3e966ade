"""GB300 (sm_103a) compressed sparse attention: a C-ABI CUDA library and its
thin Python binding.

The four calls of the path -- ``csa_compress``, ``csa_index_topk``,
``csa_sparse_attn_decode`` and ``csa_sparse_attn_prefill`` -- run entirely in
the hand-written kernels of ``libcsa.so`` (declared in ``include/csa.h``).
There is no CPU fallback: without the built library every call raises.
"""

from ._binding import (  # noqa: F401
    CSA_DEV_BAD_BLOCK,
    CSA_DEV_BAD_INDEX,
    CSA_DEV_BAD_POS,
    CSA_DEV_POS_GE_CAP,
    CSA_MODE_AUTO,
    CSA_MODE_DECODE,
    CSA_MODE_PREFILL,
    CsaError,
    csa_compress,
    csa_index_topk,
    csa_index_topk_noalloc,
    csa_sparse_attn_decode,
    csa_sparse_attn_prefill,
    launch_count,
    lib,
    prof_disable,
    prof_enable,
    prof_read,
    status_string,
    version,
)
