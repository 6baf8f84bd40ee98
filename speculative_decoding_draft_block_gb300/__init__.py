"""GB300-native draft-block sampling, confidence scheduling and lossless verification.

The hot path lives in libdsdraft.so (CUDA for sm_103a, C ABI in include/ds_draft.h).
`_lib` is its ctypes binding, `cycle.DeviceCycle` runs one cycle on device
buffers, `workloads` makes seeded synthetic inputs. Importing the package does
not load the library; the first library call does, and fails loudly if it has
not been built.
"""

__version__ = "0.1.0"
