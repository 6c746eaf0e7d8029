"""GB300-native streaming codec-to-waveform decoder (sm_103a CUDA behind a C ABI)."""
