"""Softmax-threshold block-skipping attention (BLASST) for one GB300.

The compute path is the C-ABI library ``libattn_skip.so`` built from
``csrc/``; :mod:`.binding` marshals arguments to it.  Importing this package
loads nothing; the first call into :mod:`.binding` loads the library and
raises if it is missing.
"""
__all__ = ["binding", "workloads"]
