"""ctypes access to synth/libsynth.so: fills device bf16 buffers with the
seeded generator values (same definition as the host generator)."""
import ctypes
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_PATH):
            raise ImportError(f"libsynth.so is not built ({_PATH})")
        _lib = ctypes.CDLL(_PATH)
        _lib.synth_fill_normal_bf16.restype = ctypes.c_int
        _lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong,
                                                ctypes.c_longlong, ctypes.c_void_p]
        _lib.synth_fill_e4m3.restype = ctypes.c_int
        _lib.synth_fill_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong,
                                         ctypes.c_longlong, ctypes.c_void_p]
    return _lib


def fill_normal_bf16(tensor, key: int, start: int = 0, stream=None):
    """Fill a contiguous 16-bit device tensor with values start.. of stream `key`."""
    import torch
    lib = _load()
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    err = lib.synth_fill_normal_bf16(tensor.data_ptr(), tensor.numel(), key, start, s)
    if err != 0:
        raise RuntimeError(f"synth fill failed: CUDA error {err}")


def fill_e4m3(tensor, key: int, start: int = 0, stream=None):
    """Fill a contiguous 8-bit device tensor with prefilled-pool codes start.. of stream `key`."""
    import torch
    lib = _load()
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    err = lib.synth_fill_e4m3(tensor.data_ptr(), tensor.numel(), key, start, s)
    if err != 0:
        raise RuntimeError(f"synth fill failed: CUDA error {err}")
