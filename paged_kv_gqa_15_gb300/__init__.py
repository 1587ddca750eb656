"""Paged-KV GQA attention for GB300 (sm_103a): thin binding over the C ABI."""
