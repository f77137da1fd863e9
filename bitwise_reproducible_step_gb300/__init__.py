"""GB300-native bitwise-reproducible optimizer step.

Replica gradient reduce in one canonical tree, global-norm clip over fixed 4096-element
chunks, fused AdamW over flat fp32 (w, m, v), and a chunked Merkle hash of the checkpoint
image, all as hand-written CUDA kernels for sm_103a behind the C ABI in include/repstep.h.

Submodules:
  repstep  -- the Python binding (ctypes over librepstep.so; argument marshalling only)
  inputs   -- seeded synthetic inputs (data generation only)

Importing the package loads nothing; `repstep` loads the CUDA library on first use and
raises if it is missing.
"""
