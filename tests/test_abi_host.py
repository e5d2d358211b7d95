"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol include/rlk.h declares, validates arguments before touching a device,
and its integer vocabulary-split policy depends on V only."""
import ctypes
import os
import re

import pytest
import torch

import deterministic_invariant_gemm_linear_gb300 as rlk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlk.h")

# Fake, never-dereferenced addresses: every call below fails validation first.
P16 = ctypes.c_void_p(0x10000)
NULL = None


@pytest.fixture(scope="module")
def lib():
    from deterministic_invariant_gemm_linear_gb300 import build as b
    b.build()
    return rlk.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"RLK_API\s+[^;(]*?\b(rlk_\w+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(rlk.SIGNATURES), "binding signatures must mirror the header"


def test_status_strings_and_version(lib):
    for code, name in rlk.STATUS_NAMES.items():
        assert rlk.status_string(code).startswith(name)
    assert rlk.status_string(99) == "RLK_ERR_UNKNOWN"
    m = re.search(r"#define RLK_NUMERICS_VERSION (\d+)", open(HEADER).read())
    assert rlk.numerics_version() == int(m.group(1))


@pytest.mark.parametrize("V", [1, 2, 255, 256, 257, 1024, 32003, 151936, 152064, 262144, 262145,
                               1 << 20, (1 << 31) - 257])
def test_vocab_split_policy(lib, V):
    S, vps, vt = rlk.vocab_split_policy(V)
    assert vt == -(-V // 256)
    assert 1 <= S <= 1024
    assert vps == -(-vt // 1024)
    # S contiguous, non-empty ranges covering every tile exactly once
    covered = 0
    for j in range(S):
        t0, t1 = j * vps, min((j + 1) * vps, vt)
        assert t1 > t0
        covered += t1 - t0
        assert j * vps * 256 < V                # each split holds at least one real id
    assert covered == vt


def test_vocab_split_policy_known_values(lib):
    # the configurations' vocabularies: one 256-id tile per split up to 1024 tiles
    assert rlk.vocab_split_policy(151936) == (594, 1, 594)
    assert rlk.vocab_split_policy(152064) == (594, 1, 594)
    assert rlk.vocab_split_policy(32003) == (126, 1, 126)
    assert rlk.vocab_split_policy(1024) == (4, 1, 4)
    assert rlk.vocab_split_policy(262145) == (513, 2, 1025)


def test_vocab_split_policy_rejects(lib):
    s = ctypes.c_int64()
    for V in (0, -5, 1 << 31):
        assert lib.rlk_vocab_split_policy(V, ctypes.byref(s), ctypes.byref(s), ctypes.byref(s)) == 2
    assert lib.rlk_vocab_split_policy(10, None, ctypes.byref(s), ctypes.byref(s)) == 1


def test_linear_logp_workspace_size(lib):
    f = lib.rlk_linear_logp_workspace_size
    # aligned operands: partials N*S*8 (256-aligned) + target logits N*4 (256-aligned)
    # + a 256-byte unit counter
    N, H, V = 4096, 4096, 151936
    S = 594
    want = -(-N * S * 8 // 256) * 256 + -(-N * 4 // 256) * 256 + 256
    assert f(P16, N, H, H, P16, V, H) == want
    # odd pitch of hidden: a padded copy N x 8*ceil(H/8) bf16 is added
    base = f(P16, 10, 100, 104, P16, 300, 104)
    staged = f(P16, 10, 100, 101, P16, 300, 104)
    assert staged - base == -(-(10 * 104 * 2) // 256) * 256
    # misaligned base of weight: a padded copy of W
    mis = f(ctypes.c_void_p(0x10002), 10, 100, 104, P16, 300, 104)
    assert mis - base == -(-(10 * 104 * 2) // 256) * 256
    # invalid shapes -> 0
    assert f(P16, 10, 0, 1, P16, 10, 1) == 0
    assert f(P16, 10, 8, 4, P16, 10, 8) == 0
    assert f(P16, 10, 8, 8, P16, 0, 8) == 0
    # N = 0 is valid and needs no partials (only the counter region)
    assert f(P16, 0, 8, 8, P16, 10, 8) == 256


def test_linear_logp_validation(lib):
    f = lib.rlk_linear_logp
    ws = ctypes.c_void_p(0x20000)
    # shape errors come first
    assert f(P16, 4, 0, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 2
    assert f(P16, 4, 8, 8, P16, 0, 8, NULL, P16, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 2
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, P16, -1, P16, P16, NULL, ws, 1 << 20, NULL) == 2
    # missing pointers
    assert f(NULL, 4, 8, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 1
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, NULL, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 1
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, P16, 1, NULL, P16, NULL, ws, 1 << 20, NULL) == 1
    # misaligned target / bias
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, ctypes.c_void_p(0x10004), 1, P16, P16, NULL, ws,
             1 << 20, NULL) == 4
    assert f(P16, 4, 8, 8, P16, 10, 8, ctypes.c_void_p(0x10002), P16, 1, P16, P16, NULL, ws,
             1 << 20, NULL) == 4
    # workspace missing or too small
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, NULL, 1 << 20, NULL) == 5
    assert f(P16, 4, 8, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, ws, 16, NULL) == 5
    # N == 0 is a no-op
    assert f(NULL, 0, 8, 8, NULL, 10, 8, NULL, NULL, 1, NULL, NULL, NULL, NULL, 0, NULL) == 0


def test_det_gemm_validation(lib):
    fwd, da, db = lib.rlk_det_gemm_fwd, lib.rlk_det_gemm_da, lib.rlk_det_gemm_db
    ws = ctypes.c_void_p(0x20000)
    # bad dtype / shapes / leading dims
    assert fwd(P16, 4, 8, 8, P16, 8, 8, P16, 7, 8, ws, 0, NULL) == 3
    assert fwd(P16, 4, 0, 8, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 2
    assert fwd(P16, 4, 8, 7, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 2
    assert fwd(P16, 4, 8, 8, P16, 8, 8, P16, 0, 7, ws, 0, NULL) == 2
    assert da(P16, 5, 4, 8, 8, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 3
    assert db(P16, 4, 8, 8, P16, 0, 0, 8, P16, 0, 8, ws, 0, NULL) == 2
    # null output / inputs
    assert fwd(P16, 4, 8, 8, P16, 8, 8, NULL, 0, 8, ws, 0, NULL) == 1
    assert fwd(NULL, 4, 8, 8, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 1
    # misaligned FP32 output, misaligned FP32 dC
    assert fwd(P16, 4, 8, 8, P16, 8, 8, ctypes.c_void_p(0x10002), 1, 8, ws, 0, NULL) == 4
    assert da(ctypes.c_void_p(0x10002), 1, 4, 8, 8, P16, 8, 8, P16, 0, 8, ws, 1 << 20, NULL) == 4
    # staging needed (odd pitch / FP32 dC) but no workspace
    assert fwd(P16, 4, 9, 9, P16, 8, 8, P16, 0, 8, NULL, 0, NULL) == 5
    assert da(P16, 1, 4, 8, 8, P16, 8, 8, P16, 0, 8, NULL, 0, NULL) == 5
    # M == 0 forward / dA: no-op
    assert fwd(NULL, 0, 8, 8, NULL, 8, 8, NULL, 0, 8, NULL, 0, NULL) == 0
    assert da(NULL, 0, 0, 8, 8, NULL, 8, 8, NULL, 0, 8, NULL, 0, NULL) == 0


def test_det_gemm_workspace_size(lib):
    f = lib.rlk_det_gemm_workspace_size
    # aligned BF16 operands need nothing
    assert f(0, P16, 0, 64, 64, 64, P16, 0, 64, 64, 64) == 0
    # an FP32 dC is always rounded into the workspace: M x 8*ceil(N/8) bf16
    assert f(1, P16, 1, 33, 33, 33, P16, 0, 33, 33, 40) == -(-(33 * 40 * 2) // 256) * 256
    assert f(2, P16, 0, 10, 16, 16, P16, 1, 10, 20, 20) == -(-(10 * 24 * 2) // 256) * 256
    # odd pitches stage both operands
    assert f(0, P16, 0, 3, 5, 5, P16, 0, 5, 7, 7) == 2 * 256
    # FP32 where BF16 is required, bad op -> 0
    assert f(0, P16, 1, 4, 8, 8, P16, 0, 8, 8, 8) == 0
    assert f(3, P16, 0, 4, 8, 8, P16, 0, 8, 8, 8) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported(lib):
    assert lib.rlk_device_check() == 6
    ws = ctypes.c_void_p(0x20000)
    # valid arguments: the device check is what fails, before anything launches
    assert lib.rlk_linear_logp(P16, 4, 8, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, ws,
                               1 << 20, NULL) == 6
    assert lib.rlk_det_gemm_fwd(P16, 4, 8, 8, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 6
    flags = ctypes.c_uint32(7)
    assert lib.rlk_get_device_error(NULL, ctypes.byref(flags)) == 6 and flags.value == 0


def test_binding_rejects_cpu_and_grad(lib):
    h = torch.zeros(4, 8, dtype=torch.bfloat16)
    w = torch.zeros(10, 8, dtype=torch.bfloat16)
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        rlk.linear_logp(h, w, t)
    with pytest.raises(RuntimeError, match="require grad"):
        rlk.linear_logp(h.float().requires_grad_(), w, t)
    with pytest.raises(ValueError, match="CUDA"):
        rlk.det_gemm_fwd(h, w.T)


def test_throughput_split_count(lib):
    """Occupancy-driven split count of the ablation: min(vtiles, ceil(8 * pairs / row_blocks))."""
    s = ctypes.c_int64()
    f = lib.rlk_throughput_split_count
    for N, V, sms, want in [(4096, 151936, 152, 38),      # 16 row blocks: ceil(608 / 16)
                            (16384, 152064, 152, 10),     # 64 row blocks
                            (17, 32003, 152, 126),        # one row block: every tile its own split
                            (1, 151936, 152, 594),
                            (256, 1024, 152, 4),          # capped at vtiles
                            (100000, 151936, 152, 2),     # 391 row blocks: ceil(608 / 391)
                            (200000, 151936, 152, 1),     # more row blocks than 8 * pairs
                            (256, 151936, 1, 8)]:          # one SM still counts one pair
        assert f(N, V, sms, ctypes.byref(s)) == 0, (N, V, sms)
        assert s.value == want, (N, V, sms, s.value)
    for bad in [(0, 10, 152), (10, 0, 152), (1 << 31, 10, 152), (10, 1 << 31, 152), (10, 10, -1)]:
        assert f(*bad, ctypes.byref(s)) == 2
    assert f(10, 10, 152, None) == 1


def test_det_gemm_tile_plan(lib):
    """det_gemm tiling on 152 SMs (76 pairs), in wide-tile times per pair: narrow tiles
    when all wide ones fit in half a wave; the last partial wave as half tiles (0.70
    each) in a second launch when it would fill at most half the pairs and the
    reduction is at least 16384; for a K-major right operand (dA, linear forward)
    224-wide tiles (0.93 each) when their waves cost at least 2% less."""
    FWD, DA, DB, LIN = rlk.RLK_GEMM_FWD, rlk.RLK_GEMM_DA, rlk.RLK_GEMM_DB, rlk.RLK_GEMM_LINEAR_FWD
    cases = [
        ((FWD, 4096, 4096, 4096), (256, 0, 1)),       # 256 tiles, tail 28: reduction too short
        ((DB, 4096, 4096, 4096), (256, 0, 1)),
        ((DA, 4096, 4096, 4096), (224, 0, 1)),        # 16 x 19 = 304 tiles: 4 x 0.93 < 4
        ((LIN, 4096, 4096, 4096), (224, 0, 1)),       # Y = X . W^T: the same right operand
        ((DA, 3072, 4096, 3072), (224, 0, 1)),        # 192 tiles: 3 waves; 228 of 224: 3 x 0.93
        ((DA, 3072, 3072, 4096), (256, 0, 1)),        # 144 tiles: 2 waves; 168 of 224: 3 waves
        ((DA, 8192, 4096, 8192), (256, 0, 1)),        # 512 tiles: 7 waves; 608 of 224: 8 x 0.93
        ((DA, 4096, 16384, 4096), (256, 0, 1)),       # 1024 tiles: 14 waves; 1184: 16 x 0.93
        ((FWD, 4096, 3900, 16384), (256, 28, 2)),     # tail 28 <= 38, long reduction
        ((FWD, 4096, 4096, 151936), (256, 28, 2)),    # the linear-logp backward's grad_hidden
        ((DA, 4096, 4096, 151936), (256, 28, 2)),     # split 3.70 against 224-wide 3.72
        ((FWD, 4096, 151936, 4096), (256, 0, 1)),     # 9504 tiles, tail 4: reduction too short
        ((DB, 151936, 4096, 16384), (256, 4, 2)),     # 9504 tiles, tail 4, long reduction
        ((FWD, 3072, 3072, 16384), (256, 0, 1)),      # 144 tiles: tail 68 > 38
        ((DA, 256, 4096, 4096), (128, 0, 1)),         # 16 tiles: 2 x 16 <= 76, narrow throughout
        ((FWD, 1000, 1000, 1000), (128, 0, 1)),       # 16 tiles
        ((FWD, 2560, 2048, 4096), (256, 0, 1)),       # 80 tiles: 2 x 80 > 76
        ((FWD, 4864, 4096, 65536), (256, 0, 1)),      # 19 x 16 = 304 tiles = exactly 4 waves
    ]
    for (op, rows, cols, red), want in cases:
        got = rlk.det_gemm_tile_plan(op, rows, cols, red, 152)
        assert (got["tile_cols"], got["split_blocks"], got["launches"]) == want, \
            (op, rows, cols, red, got)
    # 38 wide tiles exactly fill half the pairs: narrow throughout
    assert rlk.det_gemm_tile_plan(FWD, 9728, 256, 16384, 152)["tile_cols"] == 128
    # 77 wide tiles on 76 pairs: a last wave of one tile, split when the reduction is long
    assert rlk.det_gemm_tile_plan(FWD, 256 * 77, 256, 16384, 152) == \
        {"tile_cols": 256, "split_blocks": 1, "launches": 2}
    # an odd SM count divides into floor(sm_count / 2) pairs
    assert rlk.det_gemm_tile_plan(FWD, 4096, 4096, 16384, 151)["split_blocks"] == 256 % 75
    t, b, n = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
    f = lib.rlk_det_gemm_tile_plan
    for bad in [(FWD, 0, 10, 10, 152), (FWD, 10, 0, 10, 152), (FWD, 10, 10, 0, 152),
                (FWD, 1 << 31, 10, 10, 152), (FWD, 10, 10, 10, 1), (FWD, 10, 10, 10, 0),
                (-1, 10, 10, 10, 152), (7, 10, 10, 10, 152)]:
        assert f(*bad, ctypes.byref(t), ctypes.byref(b), ctypes.byref(n)) == 2, bad
    assert f(FWD, 10, 10, 10, 152, None, ctypes.byref(b), ctypes.byref(n)) == 1


def test_splits_workspace_size(lib):
    f = lib.rlk_linear_logp_splits_workspace_size
    g = lib.rlk_linear_logp_workspace_size
    N, H, V = 4096, 4096, 151936
    assert f(P16, N, H, H, P16, V, H, 0) == g(P16, N, H, H, P16, V, H)
    assert f(P16, N, H, H, P16, V, H, 594) == g(P16, N, H, H, P16, V, H)
    for req, S in [(38, 38), (1, 1), (5000, 594), (100, 99)]:   # vps = ceil(594/req), S = ceil(594/vps)
        want = -(-N * S * 8 // 256) * 256 + -(-N * 4 // 256) * 256 + 256
        assert f(P16, N, H, H, P16, V, H, req) == want, (req, S)
    assert f(P16, N, H, H, P16, V, H, -1) == 0


def test_extent_limits(lib):
    """Row, column and vocabulary extents stay below 2^31 - 256 (the kernels index
    them in 32-bit ints); shape errors come before any other check."""
    lim = (1 << 31) - 256
    s, v, t = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    assert lib.rlk_vocab_split_policy(lim, ctypes.byref(s), ctypes.byref(v), ctypes.byref(t)) == 2
    assert lib.rlk_vocab_split_policy(lim - 1, ctypes.byref(s), ctypes.byref(v), ctypes.byref(t)) == 0
    assert t.value == -(-(lim - 1) // 256) and s.value * v.value >= t.value
    ws = ctypes.c_void_p(0x20000)
    f = lib.rlk_linear_logp
    assert f(P16, lim, 8, 8, P16, 10, 8, NULL, P16, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 2
    assert f(P16, 4, 8, 8, P16, lim, 8, NULL, P16, 1, P16, P16, NULL, ws, 1 << 20, NULL) == 2
    assert lib.rlk_linear_logp_workspace_size(P16, lim, 8, 8, P16, 10, 8) == 0
    # (split, row block) units must number below 2^31: 2^29 rows x 1024 splits do not
    assert lib.rlk_linear_logp_workspace_size(P16, 1 << 29, 8, 8, P16, 1 << 18, 8) == 0
    assert lib.rlk_throughput_split_count(lim, 10, 152, ctypes.byref(s)) == 2
    fwd = lib.rlk_det_gemm_fwd
    assert fwd(P16, lim, 8, 8, P16, 8, 8, P16, 0, 8, ws, 0, NULL) == 2
    assert fwd(P16, 4, 8, 8, P16, lim, lim, P16, 0, lim, ws, 0, NULL) == 2


def test_two_product_backward_validates_before_any_device_use(lib):
    """rlk_det_gemm_backward / rlk_det_linear_backward check both products' outputs
    before anything launches (fail closed): fake pointers, no device touched."""
    f = lib.rlk_det_gemm_backward
    M, N, K = 64, 96, 32
    # dA misaligned for FP32, dB fine
    assert f(P16, 1, M, N, N, P16, K, K, P16, N, ctypes.c_void_p(0x10002), 1, K, P16, 1, N,
             P16, 1 << 20, None) == 4
    # dB pitch below its column count
    assert f(P16, 1, M, N, N, P16, K, K, P16, N, P16, 1, K, P16, 1, N - 1, P16, 1 << 20, None) == 2
    # an unknown output dtype
    assert f(P16, 1, M, N, N, P16, K, K, P16, N, P16, 7, K, None, 1, N, P16, 1 << 20, None) == 3
    # K = 0
    assert f(P16, 1, M, N, N, P16, 0, 1, P16, N, P16, 1, 1, P16, 1, N, P16, 1 << 20, None) == 2
    g = lib.rlk_det_linear_backward
    assert g(P16, 0, M, N, N, P16, K, K, P16, K, P16, 0, K - 1, None, 0, K, P16, 1 << 20, None) == 2
    # workspace sizes: an FP32 dC is staged once (M x 8 ceil(N/8) BF16), then a 256-byte
    # unit counter (the one-launch form of the two products); the counter alone when
    # nothing is staged
    ws = lib.rlk_det_gemm_backward_workspace_size
    assert ws(P16, 1, M, N, N, P16, K, K, P16, N) == M * N * 2 + 256
    assert ws(P16, 0, M, N, N, P16, K, K, P16, N) == 256
    assert ws(P16, 1, M, N, N, P16, 0, 1, P16, N) == 0          # invalid: K = 0
