"""W8A8 quantised mixture-of-experts layer for GB300 (sm_103a)."""
