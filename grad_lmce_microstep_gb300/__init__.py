"""Fused LM-head + softmax cross-entropy micro-step for GB300 (sm_103a).

The compute lives in the C-ABI library ``liblmce.so`` (built from ``csrc/``);
``grad_lmce_microstep_gb300.lmce`` is its thin ctypes binding.  Importing this
package loads nothing; the binding loads the library on first use and raises if
it is missing.
"""

__all__ = ["lmce", "inputs", "dp"]
