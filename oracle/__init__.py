"""CPU oracle of the MLA draft-layer forward (fp64).

TEST INFRASTRUCTURE: imported only by ``tests/``, ``__graft_entry__.smoke()``
and the CPU legs of ``bench.py``.  It shares no code with the CUDA library and
never imports it.  ``mla`` is the numpy fp64 oracle; ``brute`` is an
independent scalar-loop transcription for tiny dims; ``keys`` runs the oracle
over a paged-cache workload (which keys each block attends).

Every function of ``mla`` is pinned by ``tests/test_oracle.py`` (closed forms,
invariants, brute force, planted mutations).  Parts that rest on a reading of
the pages rather than on the pages themselves are marked there: the sliding
window edge, the interleaved output layout and the gate definition.
"""
