"""GB300-native chunkwise delta-rule token mixer (DeltaNet, Gated DeltaNet,
Kimi Delta Attention): forward and backward on one GPU through a C-ABI library
(``libdr.so``) of hand-written sm_103a kernels.

Importing the package loads nothing; the CUDA library is opened on first use by
``delta_rule_recurrent_gated_gb300.binding``.
"""
__all__ = ["binding", "inputs"]
