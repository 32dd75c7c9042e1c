"""GB300 (sm_103a) library for sample packing and document-masked causal
attention over packed rows.

The compute lives in a C-ABI shared library (``csrc/``, declared in
``include/spd.h``); ``ops`` is the thin Python binding over it. Importing the
package does not load the library; the first call into ``ops`` does, and it
raises if the library is missing or no GPU is present: there is no CPU
fallback.
"""
