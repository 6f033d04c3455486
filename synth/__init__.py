"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This package draws numbers and rounds them to the storage type; it holds none
of the block's arithmetic.
"""
from .inputs import (BlockShape, SHAPES, bf16_round, block_inputs, PARAM_NAMES,
                     attn_param_names, ffn_param_names)

__all__ = ["BlockShape", "SHAPES", "bf16_round", "block_inputs", "PARAM_NAMES",
           "attn_param_names", "ffn_param_names"]
