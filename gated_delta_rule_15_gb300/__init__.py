"""GB300-native gated delta rule: chunkwise forward and single-token decode.

The compute lives in the C-ABI library ``libdr.so`` (CUDA, sm_103a), declared in
``include/dr.h``.  ``gated_delta_rule_15_gb300.dr`` is its thin ctypes binding; importing
it loads the library and fails loudly if it has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).
"""
__all__ = ["dr", "inputs"]
