"""CPU oracle of the SRWM forward recurrence (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import this
package.  The product path (self_referential_weight_gb300) never does.
"""
from .srwm_oracle import delta_update, forward, lib_path  # noqa: F401
