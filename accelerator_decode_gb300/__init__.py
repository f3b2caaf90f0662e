"""GB300 (sm_103a) greedy decode step of a Gemma-4-E2B-shaped decoder.

    accelerator_decode_gb300/csrc/   CUDA kernels and the C ABI (libg4.so, include/g4.h)
    accelerator_decode_gb300/g4.py   ctypes binding with the C names
    accelerator_decode_gb300/runtime.py  PyTorch device-memory plumbing (Decoder, LinearOp)
    accelerator_decode_gb300/build.py    nvcc build of libg4.so

Importing the binding loads libg4.so and raises if it is missing: there is no fallback.
"""
