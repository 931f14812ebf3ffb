"""DARTree supertree construction on GB300 (sm_103a).

Importing the package loads nothing; the CUDA library is loaded on first use
by :mod:`speculative_decoding_draft_06_gb300.dartree` and raises if it has not
been built.
"""
