"""GB300 (sm_103a) flash-attention forward/backward in three numerical modes
(baseline safe softmax, stabilised safe softmax, FP32 output), behind the C ABI
in include/fa.h.  ``fa`` is the ctypes binding, ``inputs`` the seeded
workload generator, ``build`` the nvcc build of the in-tree library."""
