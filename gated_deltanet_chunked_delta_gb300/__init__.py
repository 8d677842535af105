"""GB300 (sm_103a) Gated DeltaNet chunked prefill: forward and backward."""
