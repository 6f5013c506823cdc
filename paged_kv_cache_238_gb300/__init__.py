"""GB300-native attention over a paged KV cache.

Two operations run as hand-written sm_103a CUDA kernels behind a C ABI
(``include/pa.h``, built into ``libpa.so`` inside this package):

* ``pa_reshape_and_cache`` scatters new K/V tokens into their slots of a pool of
  16-token physical blocks.
* ``pa_decode`` / ``pa_prefill_chunk`` compute decode and causal chunked-prefill
  attention, gathering K/V through an int32 block table inside the kernel.

``paged_kv_cache_238_gb300.binding`` is the thin Python layer over the C ABI
(argument marshalling only). Importing this package loads nothing; the CUDA
library is loaded on first use and its absence is an error, never a fallback.
"""

__all__ = ["binding", "workloads"]
