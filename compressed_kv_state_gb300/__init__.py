"""GB300-native Key-Value Means (KVM) layer forward.

The compute path is the C-ABI library ``libkvm.so`` (hand-written CUDA for
sm_103a); ``compressed_kv_state_gb300.kvm`` is its thin ctypes binding.  The
binding is imported lazily so that the input generators in ``workloads`` can
be used on machines without the library.
"""
__all__ = ["kvm", "workloads"]
