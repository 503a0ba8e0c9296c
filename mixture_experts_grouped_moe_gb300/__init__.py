"""GB300-native fused Mixture-of-Experts layer (sm_103a CUDA kernels behind a C ABI).

`moe` is the thin ctypes binding of the C library (`include/moe.h`); `synth`
draws seeded synthetic inputs.  Importing the package loads nothing; the
binding loads the CUDA library on first use and raises if it is missing.
"""
