"""CPU oracle of the Engram layer: test infrastructure only (tests, smoke check
and the CPU baseline of the benchmark); the product path never imports it."""
