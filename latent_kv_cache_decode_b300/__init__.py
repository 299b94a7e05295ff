"""SlimKV reconstruction-free decode attention on B300 (sm_103a).

The compute lives in ``libslimkv.so`` (hand-written CUDA behind a C ABI, see
``include/slimkv.h``); ``binding`` marshals torch tensors to it.
"""
