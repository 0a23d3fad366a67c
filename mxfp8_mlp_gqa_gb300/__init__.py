"""mxfp8_mlp_gqa_gb300: GB300 (sm_103a) CUDA kernels for one slow-AR decoder-layer
step of Dual-AR TTS decoding, behind the C-ABI library ``libmxg.so``.

``mxfp8_mlp_gqa_gb300.api`` is the Python binding (same names as the C entry
points); ``synth`` holds the seeded input generators. Importing the package
does not load the CUDA library; the first call into ``api`` does, and fails
loudly if it is missing.
"""
