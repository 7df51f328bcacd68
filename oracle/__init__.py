"""CPU oracle of the FAST-AR per-chunk attention step (test infrastructure only).

Importable by the tests, the smoke check and the benchmark's CPU-baseline arm; never
by the product path."""
