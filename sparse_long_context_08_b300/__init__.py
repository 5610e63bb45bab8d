"""EntmaxKV on B300: support-aware sparse alpha-entmax decode over a paged KV
cache, as hand-written CUDA for sm_103a behind a C ABI (include/entmaxkv.h).

Submodules:
  entmaxkv   the thin binding of the C ABI (same function names)
  api        EntmaxKVDecoder: buffers + score -> select -> decode
  workloads  seeded synthetic decode workloads (inputs only)
  build      in-tree build of libentmaxkv.so
"""

__all__ = ["entmaxkv", "api", "workloads", "build"]
