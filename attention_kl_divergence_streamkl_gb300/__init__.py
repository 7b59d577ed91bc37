"""libstreamkl: fused one-pass attention KL divergence on GB300 (sm_103a)."""
