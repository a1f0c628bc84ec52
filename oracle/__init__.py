"""CPU oracle for the eviction step. Test infrastructure only: the product path never imports it."""
