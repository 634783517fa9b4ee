"""libfattn for GB300: tiled attention, paged attention and the fused KV-cache
append behind a C ABI (include/fattn.h).  ``fattn`` is the Python binding."""
