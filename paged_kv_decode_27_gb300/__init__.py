"""GB300-native paged KV-cache decode attention.

The compute path is a C-ABI CUDA library (``include/pa.h``) built for sm_103a;
``paged_kv_decode_27_gb300.binding`` marshals torch tensors into it and
``paged_kv_decode_27_gb300.workloads`` builds seeded synthetic inputs.  The
library is loaded lazily, on the first call into the binding.
"""
