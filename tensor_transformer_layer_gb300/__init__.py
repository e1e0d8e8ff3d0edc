"""Python binding of libmptp (the C-ABI library in ``_lib/libmptp.so``).

Argument marshalling only: every function below checks the torch tensors'
dtype, shape, device and contiguity, takes their device pointers and the
current CUDA stream, and calls the C entry point of the same name. All compute
runs in the library's CUDA kernels. There is no fallback: if the library is
missing or fails to load, calls raise.

Shapes (row-major, contiguous):
  mp_mlp_fwd(X[T,h], A[h,f], B[f,h], Z[T,h], Y[T,f], U_save[T,f] | None, t)
  mp_mlp_bwd(X, A, B, U[T,f], Y[T,f], dZ[T,h], dX[T,h], dA[h,f], dB[f,h], dU_ws[T,f], t)
  mp_mlp_fwd_shards / mp_mlp_bwd_shards: the same with shard_begin, shard_count
  mp_mlp_fwd_fused / mp_mlp_bwd_fused: the same, one launch per direction, with a zeroed
      uint8 workspace of mp_mlp_fused_workspace_bytes(T, h, f, t) bytes
  mp_vocab_ce(X[T,h], E[v_pad,h], target[T] int32, loss[T] fp32, workspace uint8, v_valid, t)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmptp.so")

MP_OK = 0
MP_DEV_TIMEOUT = 0x1
MP_DEV_TARGET_RANGE = 0x2
STATUS_NAMES = {
    0: "MP_OK", 1: "MP_ERR_INVALID_ARG", 2: "MP_ERR_UNSUPPORTED_SHAPE", 3: "MP_ERR_MISALIGNED",
    4: "MP_ERR_NO_DEVICE", 5: "MP_ERR_CUDA", 6: "MP_ERR_TIMEOUT", 7: "MP_ERR_TARGET_RANGE",
    8: "MP_ERR_WORKSPACE",
}
# Every symbol include/mptp.h declares.
EXPORTS = ("mp_mlp_fwd", "mp_mlp_bwd", "mp_mlp_fwd_shards", "mp_mlp_bwd_shards", "mp_mlp_fused_workspace_bytes",
           "mp_mlp_fwd_fused", "mp_mlp_bwd_fused", "mp_vocab_ce_workspace_bytes", "mp_vocab_ce", "mp_vocab_ce_partials",
           "mp_vocab_ce_combine", "mp_status_string", "mp_status_from_device", "mp_version",
           "mp_vocab_ce_noalloc", "mp_vocab_ce_bwd_workspace_bytes", "mp_vocab_ce_bwd_workspace_bytes_one_pass",
           "mp_vocab_ce_bwd", "mp_vocab_ce_lse", "mp_vocab_ce_bwd_lse", "mp_vocab_embed",
           "mp_attn_fwd")


class MptpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = int(code)
        super().__init__(f"{fn}: {status_string(code)}")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def lib() -> ctypes.CDLL:
    """Load (once) and return the C library. Raises OSError if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"libmptp.so is not built ({LIB_PATH}); run "
                          "`python -m tensor_transformer_layer_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.mp_mlp_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]
        L.mp_mlp_fwd.restype = _I
        L.mp_mlp_bwd.argtypes = [_P] * 10 + [_I, _I, _I, _I, _P, _P]
        L.mp_mlp_bwd.restype = _I
        L.mp_mlp_fwd_shards.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]
        L.mp_mlp_fwd_shards.restype = _I
        L.mp_mlp_bwd_shards.argtypes = [_P] * 10 + [_I, _I, _I, _I, _I, _I, _P, _P]
        L.mp_mlp_bwd_shards.restype = _I
        L.mp_mlp_fused_workspace_bytes.argtypes = [_I, _I, _I, _I]
        L.mp_mlp_fused_workspace_bytes.restype = ctypes.c_size_t
        L.mp_mlp_fwd_fused.argtypes = [_P] * 6 + [_I] * 6 + [_P, ctypes.c_size_t, _P, _P]
        L.mp_mlp_fwd_fused.restype = _I
        L.mp_mlp_bwd_fused.argtypes = [_P] * 10 + [_I] * 6 + [_P, ctypes.c_size_t, _P, _P]
        L.mp_mlp_bwd_fused.restype = _I
        L.mp_vocab_ce_workspace_bytes.argtypes = [_I, _I, _I]
        L.mp_vocab_ce_workspace_bytes.restype = ctypes.c_size_t
        L.mp_vocab_ce.argtypes = [_P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce.restype = _I
        L.mp_vocab_ce_partials.argtypes = [_P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_partials.restype = _I
        L.mp_vocab_ce_combine.argtypes = [_P, ctypes.c_size_t, _P, _P, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_combine.restype = _I
        L.mp_vocab_ce_bwd_workspace_bytes.argtypes = [_I, _I, _I, _I]
        L.mp_vocab_ce_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.mp_vocab_ce_bwd_workspace_bytes_one_pass.argtypes = [_I, _I, _I, _I]
        L.mp_vocab_ce_bwd_workspace_bytes_one_pass.restype = ctypes.c_size_t
        L.mp_vocab_ce_bwd.argtypes = [_P] * 7 + [_P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_bwd.restype = _I
        L.mp_vocab_ce_lse.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_lse.restype = _I
        L.mp_vocab_ce_bwd_lse.argtypes = [_P] * 7 + [_P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_bwd_lse.restype = _I
        L.mp_attn_fwd.argtypes = [_P] * 6 + [_I, _I, _I, _I, _I, _P, _P]
        L.mp_attn_fwd.restype = _I
        L.mp_vocab_embed.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_embed.restype = _I
        L.mp_vocab_ce_noalloc.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]
        L.mp_vocab_ce_noalloc.restype = _I
        L.mp_status_string.argtypes = [_I]
        L.mp_status_string.restype = ctypes.c_char_p
        L.mp_status_from_device.argtypes = [ctypes.c_uint32]
        L.mp_status_from_device.restype = _I
        L.mp_version.argtypes = []
        L.mp_version.restype = _I
        _lib = L
    return _lib


def status_string(code: int) -> str:
    try:
        return lib().mp_status_string(int(code)).decode()
    except OSError:
        return STATUS_NAMES.get(int(code), f"status {code}")


def _ptr(x, name, dtype=torch.bfloat16, shape=None, allow_none=False):
    if x is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if x.numel() > 0 and not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return x.data_ptr() or None


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _status_ptr(d_status):
    if d_status is None:
        return None
    return _ptr(d_status, "d_status", dtype=torch.int32, shape=(1,))


def _check(fn, code):
    if code != MP_OK:
        raise MptpError(fn, code)


def mp_mlp_fwd(X, A, B, Z, Y, U_save=None, *, t: int, d_status=None, stream=None) -> None:
    """Forward of the sharded MLP: Y = GeLU(X A) (U_save = X A), Z = sum_i Y_i B_i."""
    T, h = X.shape
    f = A.shape[1]
    code = lib().mp_mlp_fwd(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(Z, "Z", shape=(T, h)), _ptr(Y, "Y", shape=(T, f)),
        _ptr(U_save, "U_save", shape=(T, f), allow_none=True),
        T, h, f, int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_fwd", code)


def mp_mlp_bwd(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, *, t: int, d_status=None, stream=None) -> None:
    """Backward of the sharded MLP: dX (shard sum fused), dA, dB; dU_ws holds dU."""
    T, h = X.shape
    f = A.shape[1]
    code = lib().mp_mlp_bwd(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(U, "U", shape=(T, f)), _ptr(Y, "Y", shape=(T, f)), _ptr(dZ, "dZ", shape=(T, h)),
        _ptr(dX, "dX", shape=(T, h)), _ptr(dA, "dA", shape=(h, f)), _ptr(dB, "dB", shape=(f, h)),
        _ptr(dU_ws, "dU_ws", shape=(T, f)), T, h, f, int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_bwd", code)


def mp_mlp_fwd_shards(X, A, B, Z, Y, U_save=None, *, t: int, shard_begin: int, shard_count: int, d_status=None,
                      stream=None) -> None:
    """Forward of shards [shard_begin, shard_begin + shard_count): their columns of Y (and
    U_save) and their partial output Z = sum over the range of Y_i B_i."""
    T, h = X.shape
    f = A.shape[1]
    code = lib().mp_mlp_fwd_shards(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(Z, "Z", shape=(T, h)), _ptr(Y, "Y", shape=(T, f)),
        _ptr(U_save, "U_save", shape=(T, f), allow_none=True),
        T, h, f, int(t), int(shard_begin), int(shard_count), _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_fwd_shards", code)


def mp_mlp_bwd_shards(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, *, t: int, shard_begin: int, shard_count: int,
                      d_status=None, stream=None) -> None:
    """Backward of shards [shard_begin, shard_begin + shard_count): their part of dX, their
    columns of dA and dU_ws, their rows of dB."""
    T, h = X.shape
    f = A.shape[1]
    code = lib().mp_mlp_bwd_shards(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(U, "U", shape=(T, f)), _ptr(Y, "Y", shape=(T, f)), _ptr(dZ, "dZ", shape=(T, h)),
        _ptr(dX, "dX", shape=(T, h)), _ptr(dA, "dA", shape=(h, f)), _ptr(dB, "dB", shape=(f, h)),
        _ptr(dU_ws, "dU_ws", shape=(T, f)), T, h, f, int(t), int(shard_begin), int(shard_count),
        _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_bwd_shards", code)


def mp_mlp_fused_workspace_bytes(T: int, h: int, f: int, t: int) -> int:
    return int(lib().mp_mlp_fused_workspace_bytes(int(T), int(h), int(f), int(t)))


def mp_mlp_fused_workspace(T: int, h: int, f: int, t: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for mp_mlp_fwd_fused / mp_mlp_bwd_fused (every call leaves it zero)."""
    return torch.zeros(mp_mlp_fused_workspace_bytes(T, h, f, t), dtype=torch.uint8, device=device)


def mp_mlp_fwd_fused(X, A, B, Z, Y, U_save=None, *, t: int, workspace, shard_begin: int = 0,
                     shard_count: int | None = None, d_status=None, stream=None) -> None:
    """mp_mlp_fwd_shards in one launch (both GEMMs of the forward); equal outputs bit for bit."""
    T, h = X.shape
    f = A.shape[1]
    n = int(t) - int(shard_begin) if shard_count is None else int(shard_count)
    wp, wb = _ws(workspace)
    code = lib().mp_mlp_fwd_fused(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(Z, "Z", shape=(T, h)), _ptr(Y, "Y", shape=(T, f)),
        _ptr(U_save, "U_save", shape=(T, f), allow_none=True),
        T, h, f, int(t), int(shard_begin), n, wp, wb, _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_fwd_fused", code)


def mp_mlp_bwd_fused(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, *, t: int, workspace, shard_begin: int = 0,
                     shard_count: int | None = None, d_status=None, stream=None) -> None:
    """mp_mlp_bwd_shards in one launch (dU, dX, dA, dB); equal outputs bit for bit."""
    T, h = X.shape
    f = A.shape[1]
    n = int(t) - int(shard_begin) if shard_count is None else int(shard_count)
    wp, wb = _ws(workspace)
    code = lib().mp_mlp_bwd_fused(
        _ptr(X, "X", shape=(T, h)), _ptr(A, "A", shape=(h, f)), _ptr(B, "B", shape=(f, h)),
        _ptr(U, "U", shape=(T, f)), _ptr(Y, "Y", shape=(T, f)), _ptr(dZ, "dZ", shape=(T, h)),
        _ptr(dX, "dX", shape=(T, h)), _ptr(dA, "dA", shape=(h, f)), _ptr(dB, "dB", shape=(f, h)),
        _ptr(dU_ws, "dU_ws", shape=(T, f)), T, h, f, int(t), int(shard_begin), n, wp, wb,
        _status_ptr(d_status), _stream(stream))
    _check("mp_mlp_bwd_fused", code)


def mp_vocab_ce_workspace_bytes(T: int, v_pad: int, t: int) -> int:
    return int(lib().mp_vocab_ce_workspace_bytes(int(T), int(v_pad), int(t)))


def _ws(workspace):
    if not isinstance(workspace, torch.Tensor) or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous torch.Tensor")
    return workspace.data_ptr() or None, workspace.numel() * workspace.element_size()


def mp_vocab_ce(X, E, target, loss, workspace, *, v_valid: int, t: int, d_status=None, stream=None) -> None:
    """Fused vocab-parallel logits + cross-entropy: loss[T] fp32."""
    T, h = X.shape
    v_pad = E.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), _ptr(loss, "loss", dtype=torch.float32, shape=(T,)),
        wp, wb, T, h, v_pad, int(v_valid), int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_ce", code)


def mp_vocab_ce_lse(X, E, target, loss, lse, workspace, *, v_valid: int, t: int, d_status=None, stream=None) -> None:
    """mp_vocab_ce that also writes the per-token log-sum-exp lse[T] fp32 (NaN for invalid targets)."""
    T, h = X.shape
    v_pad = E.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce_lse(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), _ptr(loss, "loss", dtype=torch.float32, shape=(T,)),
        _ptr(lse, "lse", dtype=torch.float32, shape=(T,)), wp, wb, T, h, v_pad, int(v_valid), int(t),
        _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_ce_lse", code)


def mp_vocab_ce_partials(X, E, target, workspace, *, v_valid: int, t: int, d_status=None, stream=None) -> None:
    T, h = X.shape
    v_pad = E.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce_partials(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), wp, wb, T, h, v_pad, int(v_valid), int(t),
        _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_ce_partials", code)


def mp_vocab_ce_combine(workspace, target, loss, *, v_pad: int, v_valid: int, t: int, d_status=None,
                        stream=None) -> None:
    T = target.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce_combine(
        wp, wb, _ptr(target, "target", dtype=torch.int32, shape=(T,)),
        _ptr(loss, "loss", dtype=torch.float32, shape=(T,)), T, int(v_pad), int(v_valid), int(t),
        _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_ce_combine", code)


def mp_vocab_ce_noalloc(X, E, target, loss, *, v_valid: int, t: int, d_status=None, stream=None) -> None:
    """mp_vocab_ce without a workspace argument, for callers that cannot allocate
    device memory: the library's fixed 4 MiB static device array holds the
    triples. Calls that overlap on the GPU race on that array."""
    T, h = X.shape
    v_pad = E.shape[0]
    code = lib().mp_vocab_ce_noalloc(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), _ptr(loss, "loss", dtype=torch.float32, shape=(T,)),
        T, h, v_pad, int(v_valid), int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_ce_noalloc", code)


def mp_vocab_ce_bwd_workspace_bytes(T: int, h: int, v_pad: int, t: int) -> int:
    return int(lib().mp_vocab_ce_bwd_workspace_bytes(int(T), int(h), int(v_pad), int(t)))


def mp_vocab_ce_bwd_workspace_bytes_one_pass(T: int, h: int, v_pad: int, t: int) -> int:
    return int(lib().mp_vocab_ce_bwd_workspace_bytes_one_pass(int(T), int(h), int(v_pad), int(t)))


def mp_vocab_ce_bwd(X, E, target, loss, dloss, dX, dE, workspace, *, v_valid: int, t: int, d_status=None,
                    stream=None) -> None:
    """Backward of the fused vocab-parallel cross-entropy: dX [T,h], dE [v_pad,h] (bf16)."""
    T, h = X.shape
    v_pad = E.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce_bwd(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), _ptr(loss, "loss", dtype=torch.float32, shape=(T,)),
        _ptr(dloss, "dloss", dtype=torch.float32, shape=(T,)), _ptr(dX, "dX", shape=(T, h)),
        _ptr(dE, "dE", shape=(v_pad, h)), wp, wb, T, h, v_pad, int(v_valid), int(t), _status_ptr(d_status),
        _stream(stream))
    _check("mp_vocab_ce_bwd", code)


def mp_vocab_ce_bwd_lse(X, E, target, lse, dloss, dX, dE, workspace, *, v_valid: int, t: int, d_status=None,
                        stream=None) -> None:
    """Backward of the fused cross-entropy from the forward's exported log-sum-exp."""
    T, h = X.shape
    v_pad = E.shape[0]
    wp, wb = _ws(workspace)
    code = lib().mp_vocab_ce_bwd_lse(
        _ptr(X, "X", shape=(T, h)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(target, "target", dtype=torch.int32, shape=(T,)), _ptr(lse, "lse", dtype=torch.float32, shape=(T,)),
        _ptr(dloss, "dloss", dtype=torch.float32, shape=(T,)), _ptr(dX, "dX", shape=(T, h)),
        _ptr(dE, "dE", shape=(v_pad, h)), wp, wb, T, h, v_pad, int(v_valid), int(t), _status_ptr(d_status),
        _stream(stream))
    _check("mp_vocab_ce_bwd_lse", code)


def mp_vocab_embed(ids, E, out, *, v_valid: int, t: int, d_status=None, stream=None) -> None:
    """Vocab-parallel embedding lookup: out[r] = E[ids[r]] (zeros for ids outside [0, v_valid))."""
    T = ids.shape[0]
    v_pad, h = E.shape
    code = lib().mp_vocab_embed(
        _ptr(ids, "ids", dtype=torch.int32, shape=(T,)), _ptr(E, "E", shape=(v_pad, h)),
        _ptr(out, "out", shape=(T, h)), T, h, v_pad, int(v_valid), int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_vocab_embed", code)


def mp_attn_fwd(X, Wqkv, Wo, out, QKV, O, *, b: int, s: int, heads: int, t: int, d_status=None,
                stream=None) -> None:
    """Head-parallel causal self-attention block: QKV = X Wqkv, per-head attention O, out = O Wo."""
    T, h = X.shape
    if T != b * s:
        raise ValueError("X must have b * s rows")
    code = lib().mp_attn_fwd(
        _ptr(X, "X", shape=(T, h)), _ptr(Wqkv, "Wqkv", shape=(h, 3 * h)), _ptr(Wo, "Wo", shape=(h, h)),
        _ptr(out, "out", shape=(T, h)), _ptr(QKV, "QKV", shape=(T, 3 * h)), _ptr(O, "O", shape=(T, h)),
        int(b), int(s), h, int(heads), int(t), _status_ptr(d_status), _stream(stream))
    _check("mp_attn_fwd", code)


def mp_status_from_device(bits: int) -> int:
    return int(lib().mp_status_from_device(ctypes.c_uint32(int(bits) & 0xFFFFFFFF)))


def mp_version() -> int:
    return int(lib().mp_version())
