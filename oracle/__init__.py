"""CPU fp64 oracle for the paged KV-cache composition.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU-baseline leg; never by the library's product path.
"""
