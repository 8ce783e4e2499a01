"""GB300-native reduce-copy and batched-copy engine.

``copy_reduce_dst_gb300.tb`` binds the CUDA library (include/tb.h):
TransferBench's GPU-executor reduce-copy ``dst = src0 + ... + srcN-1`` with
source-slice rotation, and the Mooncake-style batched descriptor copy.
``copy_reduce_dst_gb300.workloads`` generates the seeded synthetic inputs.
The binding is imported on demand so the input generators work without a
built library; importing ``tb`` without one raises ImportError.
"""
