"""GB300-native fused Gemma add-RMSNorm + FP8 / NVFP4 input quantization."""
