"""FP64 CPU oracle of the chunked Gated DeltaNet training path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / reference legs may import this package; the
product library never does, and shares no code with it.

Modules:
  gdn_oracle.c  per-token FP64 recurrence and its hand-derived reverse mode
  ref.py        ctypes binding, per-(document, q/k-head group) driver, threads
  chunked.py    the chunk-64 (WY/UT) form in FP64 numpy, forward and backward
  tables.py     brute-force enumeration of the varlen chunk tables
  conv1d.py     the short causal convolution + SiLU front, forward and backward
  kda.py        the per-channel-decay (KDA) recurrence, forward and backward
"""
