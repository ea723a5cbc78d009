"""GB300-native paged KV-cache decode attention (sm_103a).

The compute lives in the CUDA library ``libpagedkv.so`` (C ABI declared in
``include/pagedkv.h``); ``binding`` marshals torch tensors into those calls.
``inputs`` holds the seeded synthetic workload generators.  Importing the
package loads nothing; the library is loaded on first use of ``binding``.
"""

__all__ = ["binding", "inputs", "build"]
