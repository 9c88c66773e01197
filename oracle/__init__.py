"""The FastGen oracle (test infrastructure only: the tests, the smoke check
and the bench's CPU-baseline arm use it; the product never does)."""
