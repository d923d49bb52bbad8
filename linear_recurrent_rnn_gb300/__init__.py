"""librglru: the RG-LRU gated linear recurrence (Hawk / Griffin recurrent layer), forward and
backward, as hand-written CUDA kernels for GB300 (sm_103a) behind a C ABI.

``linear_recurrent_rnn_gb300.librglru`` is the thin Python binding (argument marshalling over
ctypes; every step runs in the CUDA library).  ``linear_recurrent_rnn_gb300.inputs`` draws the
seeded synthetic workloads.  Importing the package loads nothing; the shared library is loaded
on first use and a missing build raises instead of falling back to anything else.
"""
