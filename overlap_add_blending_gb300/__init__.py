"""Tiled-latent extract / trapezoid overlap-add for GB300 (sm_103a).

The compute path lives in the native library libtdp.so (C ABI in
include/tdp.h); `overlap_add_blending_gb300.tdp` is its Python binding and
raises on import when the library has not been built.  Importing the
package itself loads nothing native, so the input generators and workload
table stay usable without a GPU.
"""
