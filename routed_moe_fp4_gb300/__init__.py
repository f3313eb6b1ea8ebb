"""colimoe: a GB300-native routed MXFP4 mixture-of-experts layer behind a C ABI.

`colimoe` is the ctypes binding of libcolimoe.so (include/colimoe.h); `synthetic` draws the
seeded inputs; `build` compiles the library with nvcc for sm_103a.
"""
