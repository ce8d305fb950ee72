"""GB300 (sm_103a) sparse MLA decode: C-ABI library libsmla.so plus a thin binding.

    from sparse_mla_decode_03_gb300 import sparse_mla_decode
    out, lse = sparse_mla_decode(q, kv_cache, indices)
"""
from .api import (  # noqa: F401
    DEFAULT_SCALE, SmlaError, make_params, smla_decode_plan, smla_default_num_splits,
    smla_device_status, smla_paged_workspace_size, sparse_mla_decode_paged,
    smla_status_string, smla_workspace_size, sparse_mla_combine, sparse_mla_decode,
    sparse_mla_decode_noalloc, sparse_mla_decode_simt, sparse_mla_decode_split,
)
