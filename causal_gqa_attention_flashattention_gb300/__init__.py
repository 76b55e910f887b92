"""Causal grouped-query attention with RoPE on Q/K for GB300 (sm_103a).

The compute path is the CUDA library ``libneattn.so`` (C ABI declared in
``include/ne_attn.h``); ``binding`` marshals arguments to it.  Importing this
package does not load the library; ``binding.lib()`` does, and raises if the
library is missing.
"""
