"""fp64 CPU oracle for paged decode attention.  Test infrastructure only:
imported by the tests, the smoke check and the benchmark's CPU-baseline leg,
never by the CUDA library."""
