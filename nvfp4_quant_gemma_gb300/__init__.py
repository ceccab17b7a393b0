"""GB300-native fused Gemma add-RMSNorm + FP8 / NVFP4 input quantization.

The compute path is the sm_103a library ``libgemma_nq.so`` (C ABI declared in
``include/gemma_nq.h``); the functions below are its thin Python binding.
Importing the package does not load the library; the first call does, and
raises if the library has not been built."""
from ._binding import (  # noqa: F401
    add_rms_norm_quant,
    alloc_outputs,
    encode_e4m3_e2m1,
    gemma_add_rms_norm,
    gemma_add_rms_norm_quant,
    gemma_add_rms_norm_quant_parts,
    inject_wait_timeout,
    library_path,
    quantize_fp8_values,
    read_device_error,
    load,
    pdl_consumer,
    query_launch,
    set_launch_policy,
    set_constant_weights,
    set_pdl,
    status_string,
)
