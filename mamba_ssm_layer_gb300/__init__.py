"""GB300-native Mamba-2 layer forward: Python binding of the C-ABI library.

The heavy lifting is in ``libmamba2_gb300.so`` (CUDA kernels for sm_103a behind an
``extern "C"`` interface declared in ``include/mamba2.h``).  This package only
marshals arguments; see ``mamba_ssm_layer_gb300.abi``.
"""
