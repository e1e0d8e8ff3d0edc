"""The C-ABI library builds, loads and exports every symbol include/mptp.h declares;
argument validation answers before any CUDA work (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tensor_transformer_layer_gb300 import build
    build.build()
    import tensor_transformer_layer_gb300 as mp
    return mp.lib()


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^MP_API\s+[\w\s\*]+?\b(mp_\w+)\s*\(", src, flags=re.M)
    return names


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("mp_mlp_fwd", "mp_mlp_bwd", "mp_vocab_ce", "mp_vocab_ce_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import tensor_transformer_layer_gb300 as mp
    names = declared_symbols()
    assert sorted(names) == sorted(mp.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    import tensor_transformer_layer_gb300 as mp
    for code in range(9):
        s = mp.status_string(code)
        assert s.startswith(mp.STATUS_NAMES[code])
    assert mp.mp_status_from_device(0) == 0
    assert mp.mp_status_from_device(mp.MP_DEV_TIMEOUT) == 6
    assert mp.mp_status_from_device(mp.MP_DEV_TARGET_RANGE) == 7
    assert mp.mp_status_from_device(3) == 6
    assert mp.mp_version() >= 100


def test_workspace_bytes(L):
    import tensor_transformer_layer_gb300 as mp
    # 51,200 padded rows, t = 8: shards of 6,400 = 25 tiles of 256. T = 8192: chunks of 5 tiles,
    # P = 40 (1280 units, 17 rounds on 76 pairs either way). T = 4096: one-tile chunks, P = 200
    # (3200 units in 43 rounds of one tile, against 640 in 9 rounds of five).
    assert mp.mp_vocab_ce_workspace_bytes(8192, 51200, 8) == 40 * 3 * 8192 * 4
    assert mp.mp_vocab_ce_workspace_bytes(4096, 51200, 8) == 200 * 3 * 4096 * 4
    # v_pad / t = 384 = 3 tiles of 128: ten tokens run best as 6 one-tile chunks
    assert mp.mp_vocab_ce_workspace_bytes(10, 768, 2) == 6 * 3 * 10 * 4
    assert mp.mp_vocab_ce_workspace_bytes(10, 1000, 8) == 0     # v_pad not a multiple of 128 t
    assert mp.mp_vocab_ce_workspace_bytes(-1, 1024, 1) == 0
    assert mp.mp_vocab_ce_workspace_bytes(0, 1024, 1) == 0


def test_ce_bwd_workspace_bytes(L):
    import tensor_transformer_layer_gb300 as mp
    a256 = lambda x: (x + 255) // 256 * 256
    T, h, v_pad, t = 8192, 1536, 51200, 8
    # shard by shard: lse [T] fp32, the chain kernel's counters (64 control words, one per 256-token
    # row block and per 256-column vocabulary tile of a shard), fp32 dX accumulator [T, h], one shard
    # of dZ [T, v_pad/t] bf16
    ctr = a256(4 * (64 + 32 + 25))
    assert mp.mp_vocab_ce_bwd_workspace_bytes(T, h, v_pad, t) == (a256(T * 4) + ctr + a256(T * h * 4) +
                                                                 a256(T * 6400 * 2))
    # one pass: lse and every shard's dZ [T, v_pad] bf16
    assert mp.mp_vocab_ce_bwd_workspace_bytes_one_pass(T, h, v_pad, t) == a256(T * 4) + a256(T * v_pad * 2)
    # one shard: the two layouts coincide (no accumulator)
    assert (mp.mp_vocab_ce_bwd_workspace_bytes(300, 128, 2048, 1) ==
            mp.mp_vocab_ce_bwd_workspace_bytes_one_pass(300, 128, 2048, 1) == a256(300 * 4) + a256(300 * 2048 * 2))
    assert mp.mp_vocab_ce_bwd_workspace_bytes_one_pass(10, 64, 1000, 8) == 0   # v_pad not a multiple of 128 t


FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("T,h,f,t,code", [
    (-1, 64, 128, 1, 1),      # negative T
    (8, 0, 128, 1, 1),        # h = 0
    (8, 64, 128, 0, 1),       # t = 0
    (8, 96, 128, 1, 2),       # h % 64
    (8, 64, 192, 2, 2),       # (f/t) % 64
    (8, 64, 128, 3, 2),       # t does not divide f
])
def test_mlp_fwd_rejects_shapes(L, T, h, f, t, code):
    assert L.mp_mlp_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, T, h, f, t, None, None) == code
    assert L.mp_mlp_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, T, h, f, t, None, None) == code


@pytest.mark.parametrize("s0,n", [(-1, 1), (0, 0), (1, 2), (2, 1), (0, 3)])
def test_mlp_shards_reject_bad_ranges(L, s0, n):
    # t = 2: valid ranges are (0,1), (1,1), (0,2); anything else is MP_ERR_INVALID_ARG before any launch.
    assert L.mp_mlp_fwd_shards(FAKE, FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 2, s0, n, None, None) == 1
    assert L.mp_mlp_bwd_shards(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 2, s0, n,
                               None, None) == 1


def test_mlp_rejects_null_and_misaligned(L):
    assert L.mp_mlp_fwd(None, FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 1, None, None) == 1
    assert L.mp_mlp_fwd(FAKE, FAKE, FAKE, FAKE, None, None, 8, 64, 128, 1, None, None) == 1
    bad = ctypes.c_void_p(0x100002)
    assert L.mp_mlp_fwd(FAKE, bad, FAKE, FAKE, FAKE, None, 8, 64, 128, 1, None, None) == 3
    assert L.mp_mlp_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, bad, FAKE, 8, 64, 128, 1, None, None) == 3
    assert L.mp_mlp_bwd(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 1, None, None) == 1


def test_mlp_fused_workspace_bytes(L):
    import tensor_transformer_layer_gb300 as mp
    # 64 control words, then one counter per 256-row block and per 256-column tile of Y (dU),
    # rounded up to 256 bytes.
    a256 = lambda x: (x + 255) // 256 * 256
    assert mp.mp_mlp_fused_workspace_bytes(4096, 3072, 12288, 8) == a256(4 * (64 + 16 + 48))
    assert mp.mp_mlp_fused_workspace_bytes(300, 256, 1024, 4) == a256(4 * (64 + 2 + 4))
    assert mp.mp_mlp_fused_workspace_bytes(8, 96, 128, 1) == 0     # h % 64
    assert mp.mp_mlp_fused_workspace_bytes(8, 64, 192, 2) == 0     # (f/t) % 64


def test_mlp_fused_rejects_before_any_launch(L):
    ws = 1 << 20
    for T, h, f, t, code in ((-1, 64, 128, 1, 1), (8, 96, 128, 1, 2), (8, 64, 192, 2, 2)):
        assert L.mp_mlp_fwd_fused(FAKE, FAKE, FAKE, FAKE, FAKE, None, T, h, f, t, 0, t, FAKE, ws, None, None) == code
        assert L.mp_mlp_bwd_fused(*([FAKE] * 10), T, h, f, t, 0, t, FAKE, ws, None, None) == code
    # shard range outside [0, t)
    assert L.mp_mlp_fwd_fused(FAKE, FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 2, 1, 2, FAKE, ws, None, None) == 1
    assert L.mp_mlp_bwd_fused(*([FAKE] * 10), 8, 64, 128, 2, 2, 1, FAKE, ws, None, None) == 1
    # workspace: NULL, misaligned or smaller than mp_mlp_fused_workspace_bytes -> MP_ERR_WORKSPACE
    need = L.mp_mlp_fused_workspace_bytes(300, 256, 1024, 4)
    bad = ctypes.c_void_p(0x100004)
    for wp, wb in ((None, need), (bad, need), (FAKE, need - 4)):
        assert L.mp_mlp_fwd_fused(FAKE, FAKE, FAKE, FAKE, FAKE, None, 300, 256, 1024, 4, 0, 4, wp, wb, None,
                                  None) == 8
        assert L.mp_mlp_bwd_fused(*([FAKE] * 10), 300, 256, 1024, 4, 0, 4, wp, wb, None, None) == 8
    # T = 0 needs no workspace
    assert L.mp_mlp_fwd_fused(None, None, None, None, None, None, 0, 64, 128, 2, 0, 2, None, 0, None, None) == 0


def test_empty_batch_is_noop(L):
    assert L.mp_mlp_fwd(None, None, None, None, None, None, 0, 64, 128, 2, None, None) == 0
    assert L.mp_vocab_ce(None, None, None, None, None, 0, 0, 64, 256, 200, 2, None, None) == 0


@pytest.mark.parametrize("T,h,v_pad,v_valid,t,code", [
    (4, 64, 256, 0, 1, 1),      # v_valid < 1
    (4, 64, 256, 257, 1, 2),    # v_valid > v_pad
    (4, 64, 384, 300, 2, 2),    # v_pad % (128 t)
    (4, 32, 256, 200, 1, 2),    # h % 64
    (4, 64, 256, 200, 0, 1),    # t = 0
])
def test_ce_rejects_shapes(L, T, h, v_pad, v_valid, t, code):
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, T, h, v_pad, v_valid, t, None, None) == code


def test_ce_rejects_small_workspace_and_misaligned(L):
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, 64, 256, 200, 1, None, None) == 8
    bad = ctypes.c_void_p(0x100004)
    assert L.mp_vocab_ce(FAKE, FAKE, bad, FAKE, FAKE, 1 << 30, 4, 64, 256, 200, 1, None, None) == 3
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, None, 1 << 30, 4, 64, 256, 200, 1, None, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_no_device_answer(L):
    # Valid arguments on a machine without a GB300: MP_ERR_NO_DEVICE, nothing launched.
    assert L.mp_mlp_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 1, None, None) == 4
    assert L.mp_mlp_fwd_fused(FAKE, FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 1, 0, 1, FAKE, 1 << 20, None,
                              None) == 4
    assert L.mp_mlp_bwd_fused(*([FAKE] * 10), 8, 64, 128, 1, 0, 1, FAKE, 1 << 20, None, None) == 4
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, 4, 64, 256, 200, 1, None, None) == 4
    # The no-allocation entry point: a T = 0 call also reaches the device (it places the static
    # array there), so without one it answers MP_ERR_NO_DEVICE; a problem whose triples fit the
    # 4 MiB array in no partition (one per shard: 8 x 3 x 43,691 floats) is refused first.
    assert L.mp_vocab_ce_noalloc(None, None, None, None, 0, 64, 256, 200, 1, None, None) == 4
    assert L.mp_vocab_ce_noalloc(FAKE, FAKE, FAKE, FAKE, 43690, 64, 51200, 50257, 8, None, None) == 4
    assert L.mp_vocab_ce_noalloc(FAKE, FAKE, FAKE, FAKE, 43691, 64, 51200, 50257, 8, None, None) == 8
    # A smaller workspace than mp_vocab_ce_workspace_bytes runs a coarser partition that fits it
    # (then the device check answers); none fits: MP_ERR_WORKSPACE before any device call.
    want = 200 * 3 * 4096 * 4
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, want, 4096, 64, 51200, 50257, 8, None, None) == 4
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 4 << 20, 4096, 64, 51200, 50257, 8, None, None) == 4
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 8 * 3 * 4096 * 4, 4096, 64, 51200, 50257, 8, None,
                         None) == 4
    assert L.mp_vocab_ce(FAKE, FAKE, FAKE, FAKE, FAKE, 8 * 3 * 4096 * 4 - 4, 4096, 64, 51200, 50257, 8, None,
                         None) == 8


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import tensor_transformer_layer_gb300 as mp
    monkeypatch.setattr(mp, "_lib", None)
    monkeypatch.setattr(mp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(OSError):
        mp.lib()
