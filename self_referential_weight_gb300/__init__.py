"""GB300-native forward recurrence of the multi-head Self-Referential Weight Matrix.

The compute path is the C-ABI library libsrwm.so (hand-written sm_103a CUDA).
This package is its thin Python binding: `srwm_forward`, `srwm_step` and
`srwm_status_string` marshal torch CUDA tensors into the C calls of the same
names.  `inputs` holds the seeded synthetic workloads.  The binding is loaded
on first use, so `import self_referential_weight_gb300.inputs` needs no GPU.
"""

__all__ = ["srwm_forward", "srwm_forward_balanced", "srwm_forward_workspace_bytes", "srwm_forward_from", "srwm_step", "srwm_status_string", "SrwmError", "library_path"]


def __getattr__(name):
    if name in __all__:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
