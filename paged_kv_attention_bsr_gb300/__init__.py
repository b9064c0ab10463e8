"""Attention over a block-sparse-row (BSR) paged KV cache on one GB300 (sm_103a).

The compute path is libattn.so (C ABI in include/attn.h): a host planner that
balances work units over a persistent grid, a batch-decode kernel, a
tcgen05 append / prefill kernel and LSE merge kernels. This package is the
thin Python binding over it:

  * ``_capi``  -- ctypes marshalling, one function per C entry point;
  * ``api``    -- workspace ownership (PagedAttention), composable shared-prefix
                  decode (CascadeAttention), the single-request decode of the
                  quick-start snippet, merge_state;
  * ``synth``  -- seeded synthetic inputs (no attention arithmetic);
  * ``build``  -- nvcc build of libattn.so for sm_103a.

Importing the binding raises ImportError if libattn.so has not been built;
there is no CPU or PyTorch fallback.
"""

__all__ = ["PagedAttention", "CascadeAttention", "single_decode_with_kv_cache", "merge_state",
           "AttnError"]


def __getattr__(name):
    if name in ("PagedAttention", "CascadeAttention", "single_decode_with_kv_cache",
                "merge_state"):
        from . import api
        return getattr(api, name)
    if name == "AttnError":
        from . import _capi
        return _capi.AttnError
    raise AttributeError(name)
