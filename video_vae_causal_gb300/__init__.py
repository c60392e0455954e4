"""GB300-native Wan 2.2 VAE decoder ResidualBlock (NDHWC bf16, sm_103a)."""
