"""GB300 (sm_103a) speculative-decoding block verification.

The verify round lives in libsv.so (C ABI: include/sv.h); `binding` is its
ctypes front end and `synth` the seeded synthetic-input generators.  Import
`speculative_decoding_verification_sv_gb300.binding` to use the kernels (it
raises if the library has not been built).
"""
__all__ = ["binding", "synth", "build"]
