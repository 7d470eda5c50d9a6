"""Split-KV attention for GB300 (sm_103a): LPT-planned KV shards, partial attention, exact merge.

The compute lives in ``libsplitkv.so`` (C ABI, include/splitkv.h), built from
``csrc/`` by ``build.py``.  ``splitkv`` is its ctypes binding, ``runner`` strings
the calls together for a batch, ``workloads`` draws seeded synthetic inputs.
The library is loaded on first use, so importing the package needs no GPU.
"""

__all__ = ["splitkv", "runner", "workloads", "build"]
