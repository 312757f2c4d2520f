"""Rotated INT2 KV cache (append + mixed INT2/BF16 decode attention) for GB300.

The compute path is the C-ABI library liboscar_kv.so (hand-written CUDA for
sm_103a); ``oscar_kv`` is its thin Python binding.
"""
