"""GB300-native paged KV-cache attention.

`pagedattn` is the Python binding of the C-ABI library (libpagedattn.so):
`reshape_and_cache` and `paged_attention`.  `workloads` builds seeded
synthetic inputs.  Importing the package itself loads nothing native.
"""
__all__ = ["pagedattn", "workloads"]
