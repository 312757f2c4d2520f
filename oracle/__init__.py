"""CPU oracle — test infrastructure only (tests, smoke check, benchmark CPU baseline)."""
