"""kinv: a batch-invariant LLM forward step for GB300 (sm_103a).

The compute path is the C-ABI library ``libkinv.so`` built from ``csrc/``;
``kinv`` is its thin ctypes binding and ``model`` the decoder drivers built on
it.  Importing this package does not load the library; the first call into
``kinv`` does, and raises if it has not been built.
"""
__all__ = ["kinv", "model", "synth", "build"]
