"""GPU-resident prioritized experience replay for GB300 (sm_103a)."""
