"""GB300-native fused compressed-optimizer step (FlashAdamW, FlashSGD, FlashLion).

The hot path lives in the C-ABI library ``libfo.so`` (hand-written sm_103a CUDA,
declared in ``include/fo.h``); :mod:`quantized_optimizer_state_gb300.fo` is its
thin ctypes binding. The library is loaded on first use, and a missing or
unbuildable library raises an error: there is no CPU fallback.
"""
