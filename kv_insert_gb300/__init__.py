"""GB300-native decode-batch QKV front: projection + q/k RMS norm + interleaved
RoPE + paged K/V insert in one sm_103a kernel, behind a C ABI."""
