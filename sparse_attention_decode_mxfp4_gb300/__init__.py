"""Sparse MXFP4 attention decode step for GB300 (sm_103a).

The compute path is the C-ABI library ``libsmx.so`` (hand-written CUDA kernels); ``ops``
is its thin ctypes binding and ``workloads`` draws the seeded synthetic inputs. Importing the
package never loads the library; the first op call does, and fails loudly if it is missing.
"""
