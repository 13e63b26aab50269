"""GB300-native block-wise diffusion-LLM decoding (dual KV cache, fused LM head + threshold commit).

The compute path is the CUDA library ``libdinfer.so`` (built by ``build.py``)
behind the C-ABI declared in ``include/dinfer.h``; ``block_denoising_gb300.dinfer``
is its thin ctypes binding.  ``inputs`` holds the seeded synthetic inputs.
"""
