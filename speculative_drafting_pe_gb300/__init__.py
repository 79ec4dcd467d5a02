"""P-EAGLE parallel drafting + verify/rebuild on GB300 (sm_103a).

The compute path is the CUDA library ``libpe.so`` (C ABI declared in
``include/pe.h``); ``binding`` is a thin ctypes layer over it. Importing this
package does not load the library; ``binding.load()`` does, and fails loudly
if it is missing.
"""

__all__ = ["synth", "binding"]
