"""rs_decode_gb300: the ReplaySSM decode path as a C-ABI CUDA library (librs.so)
for GB300 (sm_103a), with a thin Python binding.

* ``binding``  ctypes binding, one function per C entry point of include/rs.h
* ``layer``    owner of one layer's state tensors (allocation via torch)
* ``synth``    seeded synthetic inputs shared by tests, benchmark and oracle
* ``build``    nvcc build of librs.so
"""
