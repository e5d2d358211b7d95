"""Guard-band canaries around every output and workspace buffer (sanitizer substitute).

Each call below writes into the middle of a larger buffer pre-filled with a
canary pattern: bytes before and after each output, the padding columns of a
pitched output, the workspace's bytes past its documented size, and the unused
slack between its 256-byte-aligned regions must all keep the canary.  Used by
tests/test_gpu_guard_bands.py with the release library in-process and with the
debug library (store checks compiled in) in a child process.
"""
import ctypes
import itertools

import torch

import deterministic_invariant_gemm_linear_gb300 as rlk
import seeded_inputs as si

CANARY_BYTE = 0xA5
GUARD = 1024                      # bytes of canary on each side of every buffer


class Guarded:
    """A device buffer of `nbytes` (plus optional row padding) with canary bands."""

    def __init__(self, nbytes: int, dev, align: int = 256):
        self.nbytes = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), CANARY_BYTE, dtype=torch.uint8, device=dev)
        assert self.raw.data_ptr() % align == 0 and GUARD % align == 0

    @property
    def ptr(self):
        return ctypes.c_void_p(self.raw.data_ptr() + GUARD)

    def body(self):
        return self.raw[GUARD:GUARD + self.nbytes]

    def bands_intact(self) -> bool:
        return bool((self.raw[:GUARD] == CANARY_BYTE).all()) and \
            bool((self.raw[GUARD + self.nbytes:] == CANARY_BYTE).all())

    def untouched(self, lo: int, hi: int) -> bool:
        """Body bytes [lo, hi) still hold the canary."""
        return hi <= lo or bool((self.body()[lo:hi] == CANARY_BYTE).all())


def _pitched_untouched(g: Guarded, rows: int, cols: int, ld: int, esize: int) -> bool:
    """The padding columns [cols, ld) of every row of a pitched output kept the canary."""
    if ld == cols or rows == 0:
        return True
    body = g.body()[:rows * ld * esize].view(rows, ld * esize)
    return bool((body[:, cols * esize:] == CANARY_BYTE).all())


def _a256(x: int) -> int:
    return -(-x // 256) * 256


def _tma_ready(t: torch.Tensor, ld: int) -> bool:
    return t.data_ptr() % 16 == 0 and ld % 8 == 0


def _staged_slack_ok(ws: Guarded, off: int, staged, ncols: int) -> bool:
    """Regions of padded copies from `off` on, in order: each [rows, 8*ceil(cols/8)] BF16
    copy is written in full and the slack up to its 256-byte boundary is not.
    staged: [(is_staged, rows)].  Returns whether every slack kept the canary and the
    regions end exactly at the workspace size."""
    ldst = -(-ncols // 8) * 8
    ok = True
    for is_staged, rows in staged:
        if not is_staged:
            continue
        used = rows * ldst * 2
        ok = ok and ws.untouched(off + used, off + _a256(used))
        off += _a256(used)
    return ok and off == ws.nbytes


def linear_logp_cases(dev, fails):
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    for N, H, V in itertools.product((1, 33, 129), (1, 8, 100), (1, 257, 32003)):
        hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=N + H + V,
                                                             device=dev)
        for odd in (False, True):
            if odd and H == 1:
                continue
            h = hidden
            if odd:                       # odd pitch: staged through the workspace
                h = torch.zeros(N, H + 1, dtype=torch.bfloat16, device=dev)
                h[:, :H] = hidden
                h = h[:, :H]
            ldh = h.stride(0)
            what = f"linear_logp N={N} H={H} V={V}{' staged hidden' if odd else ''}"
            ws_n = lib.rlk_linear_logp_workspace_size(P(h), N, H, ldh, P(weight), V, H)
            outs = [Guarded(4 * N, dev) for _ in range(3)]
            ws = Guarded(ws_n, dev)
            st = lib.rlk_linear_logp(P(h), N, H, ldh, P(weight), V, H, P(bias), P(target), 1,
                                     outs[0].ptr, outs[1].ptr, outs[2].ptr, ws.ptr, ws_n, sp)
            torch.cuda.synchronize()
            if st != 0:
                fails.append(f"{what}: status {st}")
                continue
            S = rlk.vocab_split_policy(V)[0]
            off_zt = _a256(N * S * 8)
            off_ctr = _a256(off_zt + 4 * N)
            ok = all(o.bands_intact() for o in outs) and ws.bands_intact()
            ok = ok and ws.untouched(N * S * 8, off_zt) and ws.untouched(off_zt + 4 * N, off_ctr)
            ok = ok and ws.untouched(off_ctr + 4, off_ctr + 256)
            ok = ok and _staged_slack_ok(ws, off_ctr + 256, [(not _tma_ready(h, ldh), N),
                                                             (not _tma_ready(weight, H), V)], H)
            if not ok:
                fails.append(f"{what}: a canary was overwritten")


def backward_cases(dev, fails):
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    for N, H, V in itertools.product((1, 33, 129), (1, 8, 100), (1, 257, 32003)):
        hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=N * H + V,
                                                             device=dev)
        lse = rlk.linear_logp(hidden, weight, target, bias)[1]
        g = torch.randn(N, generator=torch.Generator(device=dev).manual_seed(N), device=dev)
        for dtype, esize in ((rlk.RLK_FP32, 4), (rlk.RLK_BF16, 2)):
            what = f"backward N={N} H={H} V={V} {'fp32' if esize == 4 else 'bf16'}"
            ldh_out, ldw_out = H + 3, H + 5           # pitched outputs: padding must stay
            gh = Guarded(N * ldh_out * esize, dev)
            gw = Guarded(V * ldw_out * esize, dev)
            gb = Guarded(4 * V, dev)
            ws_n = lib.rlk_linear_logp_backward_workspace_size_for(P(hidden), N, H, H, P(weight), V,
                                                                   H)
            ws = Guarded(ws_n, dev)
            st = lib.rlk_linear_logp_backward(P(hidden), N, H, H, P(weight), V, H, P(bias),
                                              P(target), 1, P(lse), P(g), gh.ptr, dtype, ldh_out,
                                              gw.ptr, dtype, ldw_out, gb.ptr, ws.ptr, ws_n, sp)
            torch.cuda.synchronize()
            if st != 0:
                fails.append(f"{what}: status {st}")
                continue
            ldG = -(-V // 8) * 8
            off_ctr = _a256(N * ldG * 2)
            ok = gh.bands_intact() and gw.bands_intact() and gb.bands_intact() and ws.bands_intact()
            ok = ok and _pitched_untouched(gh, N, H, ldh_out, esize)
            ok = ok and _pitched_untouched(gw, V, H, ldw_out, esize)
            ok = ok and ws.untouched(N * ldG * 2, off_ctr) and ws.untouched(off_ctr + 4, off_ctr + 256)
            ok = ok and _staged_slack_ok(ws, off_ctr + 256, [(not _tma_ready(hidden, H), N),
                                                             (not _tma_ready(weight, H), V)], H)
            if not ok:
                fails.append(f"{what}: a canary was overwritten")


def det_gemm_cases(dev, fails):
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    for M, K, N in ((1, 1, 1), (33, 8, 100), (129, 100, 257), (300, 64, 33)):
        A, B, dC = si.det_gemm_inputs(M, K, N, seed=M + K + N, device=dev)
        dC32 = dC.float()
        for dtype, esize in ((rlk.RLK_FP32, 4), (rlk.RLK_BF16, 2)):
            for op in ("fwd", "da", "db"):
                rows, cols = {"fwd": (M, N), "da": (M, K), "db": (K, N)}[op]
                ld = cols + 5
                C = Guarded(rows * ld * esize, dev)
                # inputs in argument order (an FP32 dC is rounded to BF16 in the workspace)
                x, xdt, xr, xc, y, ydt, yr, yc, code = {
                    "fwd": (A, 0, M, K, B, 0, K, N, rlk.RLK_GEMM_FWD),
                    "da": (dC32, 1, M, N, B, 0, K, N, rlk.RLK_GEMM_DA),
                    "db": (A, 0, M, K, dC32, 1, M, N, rlk.RLK_GEMM_DB)}[op]
                ws_n = lib.rlk_det_gemm_workspace_size(code, P(x), xdt, xr, xc, xc, P(y), ydt, yr,
                                                       yc, yc)
                ws = Guarded(max(ws_n, 0), dev)
                if op == "fwd":
                    st = lib.rlk_det_gemm_fwd(P(A), M, K, K, P(B), N, N, C.ptr, dtype, ld, ws.ptr,
                                              ws_n, sp)
                elif op == "da":
                    st = lib.rlk_det_gemm_da(P(dC32), rlk.RLK_FP32, M, N, N, P(B), K, N, C.ptr,
                                             dtype, ld, ws.ptr, ws_n, sp)
                else:
                    st = lib.rlk_det_gemm_db(P(A), M, K, K, P(dC32), rlk.RLK_FP32, N, N, C.ptr,
                                             dtype, ld, ws.ptr, ws_n, sp)
                torch.cuda.synchronize()
                what = f"det_gemm {op} M={M} K={K} N={N} esize={esize}"
                # staged copies: x then y, each [rows, 8*ceil(cols/8)] and 256-aligned
                ok = True
                off = 0
                for t, dt, r, c in ((x, xdt, xr, xc), (y, ydt, yr, yc)):
                    if dt == 1 or not _tma_ready(t, c):
                        used = r * (-(-c // 8) * 8) * 2
                        ok = ok and ws.untouched(off + used, off + _a256(used))
                        off += _a256(used)
                ok = ok and off == ws_n and ws.bands_intact()
                if st != 0:
                    fails.append(f"{what}: status {st}")
                elif not (ok and C.bands_intact() and _pitched_untouched(C, rows, cols, ld, esize)):
                    fails.append(f"{what}: a canary was overwritten")


def det_gemm_split_cases(dev, fails):
    """Products whose last wave runs as 128-wide halves in a second launch (16 x 16
    wide tiles, reduction 16384): the halves, including the empty second half of a
    60-column last block, write only their own columns of a pitched output."""
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    R = 16384
    g = torch.Generator(device=dev).manual_seed(77)

    def bf(r, c):
        return torch.randn(r, c, generator=g, device=dev).to(torch.bfloat16)

    A, B = bf(4096, R), bf(R, 3900)          # fwd -> [4096, 3900]
    dC, Bt = bf(4096, R), bf(4000, R)        # dA = dC . Bt^T -> [4096, 4000]
    A2, dC2 = bf(R, 4000), bf(R, 3900)       # dB = A2^T . dC2 -> [4000, 3900]
    # (the 3900-column operands have an odd pitch and are staged through the workspace)
    ops = {"fwd": (4096, 3900, (rlk.RLK_GEMM_FWD, A, 4096, R, B, R, 3900)),
           "da": (4096, 4000, (rlk.RLK_GEMM_DA, dC, 4096, R, Bt, 4000, R)),
           "db": (4000, 3900, (rlk.RLK_GEMM_DB, A2, R, 4000, dC2, R, 3900))}
    for dtype, esize in ((rlk.RLK_FP32, 4), (rlk.RLK_BF16, 2)):
        for op, (rows, cols, (code, x, xr, xc, y, yr, yc)) in ops.items():
            ld = cols + 5
            C = Guarded(rows * ld * esize, dev)
            ws_n = lib.rlk_det_gemm_workspace_size(code, P(x), 0, xr, xc, xc, P(y), 0, yr, yc, yc)
            ws = Guarded(max(ws_n, 0), dev)
            if op == "fwd":
                st = lib.rlk_det_gemm_fwd(P(A), 4096, R, R, P(B), 3900, 3900, C.ptr, dtype, ld,
                                          ws.ptr, ws_n, sp)
            elif op == "da":
                st = lib.rlk_det_gemm_da(P(dC), rlk.RLK_BF16, 4096, R, R, P(Bt), 4000, R, C.ptr,
                                         dtype, ld, ws.ptr, ws_n, sp)
            else:
                st = lib.rlk_det_gemm_db(P(A2), R, 4000, 4000, P(dC2), rlk.RLK_BF16, 3900, 3900,
                                         C.ptr, dtype, ld, ws.ptr, ws_n, sp)
            torch.cuda.synchronize()
            what = f"det_gemm {op} split last wave esize={esize}"
            if st != 0:
                fails.append(f"{what}: status {st}")
            elif not (C.bands_intact() and _pitched_untouched(C, rows, cols, ld, esize) and
                      ws.bands_intact()):
                fails.append(f"{what}: a canary was overwritten")


def det_gemm_mid_width_cases(dev, fails):
    """dA and the linear forward on 256 x 224 tiles (a 4096 x 4000 output: 16 x 18
    tiles, the last column block 192 wide) write only their own columns of a pitched
    output."""
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    g = torch.Generator(device=dev).manual_seed(78)

    def bf(r, c):
        return torch.randn(r, c, generator=g, device=dev).to(torch.bfloat16)

    dC, B = bf(4096, 4096), bf(4000, 4096)   # dA = dC . B^T -> [4096, 4000]
    X, W = bf(4096, 4096), bf(4000, 4096)    # Y = X . W^T -> [4096, 4000]
    for dtype, esize in ((rlk.RLK_FP32, 4), (rlk.RLK_BF16, 2)):
        for op in ("da", "linear"):
            rows, cols = 4096, 4000
            ld = cols + 5
            C = Guarded(rows * ld * esize, dev)
            if op == "da":
                st = lib.rlk_det_gemm_da(P(dC), rlk.RLK_BF16, 4096, 4096, 4096, P(B), 4000, 4096,
                                         C.ptr, dtype, ld, None, 0, sp)
            else:
                st = lib.rlk_det_linear_fwd(P(X), 4096, 4096, 4096, P(W), 4000, 4096, C.ptr, dtype,
                                            ld, None, 0, sp)
            torch.cuda.synchronize()
            what = f"det_gemm {op} 224-wide tiles esize={esize}"
            if st != 0:
                fails.append(f"{what}: status {st}")
            elif not (C.bands_intact() and _pitched_untouched(C, rows, cols, ld, esize)):
                fails.append(f"{what}: a canary was overwritten")


def shard_cases(dev, fails):
    lib, P = rlk.lib(), rlk._ptr
    sp = rlk._stream_ptr(None)
    N, H, V = 33, 100, 32003
    hidden, weight, bias, target = si.linear_logp_inputs(N, H, V, bias=True, seed=9, device=dev)
    S, vps, _ = rlk.vocab_split_policy(V)
    for j0, j1 in ((0, 1), (3, 60), (100, S)):
        v0, v1 = j0 * vps * 256, min(j1 * vps * 256, V)
        w, b = weight[v0:v1].contiguous(), bias[v0:v1].contiguous()
        ld = j1 - j0 + 3
        parts = Guarded(N * ld * 8, dev)
        zt = Guarded(4 * N, dev)
        ws_n = lib.rlk_linear_logp_shard_workspace_size(P(hidden), N, H, H, P(w), V, j0, j1, H)
        ws = Guarded(ws_n, dev)
        st = lib.rlk_linear_logp_shard_partials(P(hidden), N, H, H, P(w), V, j0, j1, H, P(b),
                                                P(target), 1, parts.ptr, ld, zt.ptr, ws.ptr, ws_n, sp)
        torch.cuda.synchronize()
        what = f"shard partials splits [{j0}, {j1})"
        if st != 0:
            fails.append(f"{what}: status {st}")
            continue
        held = ((target >= v0) & (target < v1)).cpu()
        zb = zt.body().view(N, 4).cpu()
        ok = parts.bands_intact() and zt.bands_intact() and ws.bands_intact()
        ok = ok and _pitched_untouched(parts, N, (j1 - j0) * 8, ld * 8, 1)
        ok = ok and bool((zb[~held] == CANARY_BYTE).all()) and ws.untouched(4, 256)
        ok = ok and _staged_slack_ok(ws, 256, [(not _tma_ready(hidden, H), N),
                                               (not _tma_ready(w, H), v1 - v0)], H)
        if not ok:
            fails.append(f"{what}: a canary was overwritten")


def run_all(dev):
    fails = []
    linear_logp_cases(dev, fails)
    backward_cases(dev, fails)
    det_gemm_cases(dev, fails)
    det_gemm_split_cases(dev, fails)
    det_gemm_mid_width_cases(dev, fails)
    shard_cases(dev, fails)
    return fails
