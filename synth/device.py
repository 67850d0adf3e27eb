"""Device half of the seeded input generator: builds and wraps synth.cu.

Fills device buffers with the same values as the host generator in
``synth/__init__.py`` (same counter-based SplitMix64 definition), so that
multi-GiB benchmark inputs never pass through the host.  Also wraps the
benchmark's read-only HBM stream probe.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "synth.cu")
LIB = os.path.join(HERE, "libpirsynth.so")
COEFF, WORD, RESIDUE = 0, 1, 2


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-o", tmp, SRC])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libpirsynth.so not built: run synth.device.build()")
        L = ctypes.CDLL(LIB)
        L.synth_fill.restype = ctypes.c_int
        L.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                 ctypes.c_uint32, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                                 ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
        L.synth_fill_bytes.restype = ctypes.c_int
        L.synth_fill_bytes.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_uint32, ctypes.c_void_p]
        L.synth_read_probe.restype = ctypes.c_int
        L.synth_read_probe.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        _lib = L
    return _lib


def _stream(stream):
    import torch
    return (stream or torch.cuda.current_stream()).cuda_stream


def fill_coeffs(t, seed, tid, idx0=0, stream=None):
    rc = lib().synth_fill(t.data_ptr(), t.numel(), idx0, seed, tid, COEFF, 0, 0, None, _stream(stream))
    assert rc == 0, rc


def fill_words(t, seed, tid, idx0=0, stream=None):
    rc = lib().synth_fill(t.data_ptr(), t.numel(), idx0, seed, tid, WORD, 0, 0, None, _stream(stream))
    assert rc == 0, rc


def fill_residues(t, seed, tid, N, qs, idx0=0, stream=None):
    qa = (ctypes.c_uint32 * len(qs))(*qs)
    rc = lib().synth_fill(t.data_ptr(), t.numel(), idx0, seed, tid, RESIDUE, N, len(qs), qa, _stream(stream))
    assert rc == 0, rc


def fill_bytes(t, seed, tid, idx0=0, stream=None):
    rc = lib().synth_fill_bytes(t.data_ptr(), t.numel(), idx0, seed, tid, _stream(stream))
    assert rc == 0, rc


def read_probe(t, sink, stream=None):
    """One read-only pass over the bytes of device tensor t (sink: 1 int32 on the device)."""
    rc = lib().synth_read_probe(t.data_ptr(), t.numel() * t.element_size() // 16 * 16, sink.data_ptr(),
                                _stream(stream))
    assert rc == 0, rc
