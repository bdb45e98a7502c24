"""B300-native selective state-space scan (Mamba-1 selective SSM): prefill scan and one-token decode.

The compute runs in hand-written CUDA kernels for sm_103a behind a C ABI (``include/ssm.h``);
``selective_state_space_139_b300.ssm`` is a thin ctypes binding over that library.
"""
__all__ = ["workloads"]
