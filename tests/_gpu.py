"""Helpers for the GPU parity tests: guarded device buffers and a checked run.

Every device buffer sits inside a larger allocation whose surrounding bytes
(4 KiB before and after) hold a canary; outputs also get a few rows of
sentinel-filled slack past the rows they receive.  ``run_and_check`` runs the
exchange through the C ABI (the Python binding), then checks, against the CPU
oracle: every output byte, out_splits_offsets, that canaries and slack are
untouched, and that the inputs were not modified.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import variable_size_all_gb300 as a2av

GUARD = 4096
CANARY = 0xA5
SENTINEL = 0xEE
SLACK_ROWS = 3


class Guarded:
    """A device view of ``nbytes`` bytes at ``mis`` bytes past a 4 KiB boundary."""

    def __init__(self, nbytes: int, mis: int = 0, fill: int = CANARY, host=None):
        self.nbytes, self.mis = int(nbytes), int(mis)
        self.full = torch.full((GUARD + self.mis + self.nbytes + GUARD,), CANARY,
                               dtype=torch.uint8, device="cuda")
        self.view = self.full[GUARD + self.mis: GUARD + self.mis + self.nbytes]
        if host is not None:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(host)))
        elif fill != CANARY:
            self.view.fill_(fill)

    def guards_intact(self) -> bool:
        f = self.full.cpu().numpy()
        lo, hi = GUARD + self.mis, GUARD + self.mis + self.nbytes
        return bool(np.all(f[:lo] == CANARY) and np.all(f[hi:] == CANARY))


def exchange_checked(inputs, S, rb, path=a2av.PATH_AUTO, in_mis=None, out_mis=None,
                     ctas_per_sm=0, stream=None, engine=None, expect_path=None):
    """Run one exchange on the GPU and compare everything with the oracle."""
    W = len(inputs)
    S = np.ascontiguousarray(S, dtype=np.int64)
    in_mis = in_mis or [0] * W
    out_mis = out_mis or [0] * W
    recv = [int(S[:, p].sum()) for p in range(W)]
    ins = [Guarded(inputs[r].size, in_mis[r], host=inputs[r]) for r in range(W)]
    outs = [Guarded((recv[p] + SLACK_ROWS) * rb, out_mis[p], fill=SENTINEL) for p in range(W)]
    splits = torch.from_numpy(S).cuda()
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    own = engine is None
    eng = engine or a2av.A2av(W, path=path, ctas_per_sm=ctas_per_sm)
    try:
        eng.run([g.view for g in ins], splits, [g.view for g in outs], so, rb, stream=stream)
        st = eng.status(stream)
        launch = eng.last_launch()
    finally:
        if own:
            eng.close()
    torch.cuda.synchronize()
    assert st == a2av.OK, f"device status {st}"
    if expect_path is not None:
        assert launch["path"] == expect_path, launch
    ref, ref_so = oracle.default().exchange(inputs, S, rb)
    assert np.array_equal(so.cpu().numpy(), ref_so), "out_splits_offsets differ from the oracle"
    for p in range(W):
        got = outs[p].view.cpu().numpy()
        n = recv[p] * rb
        if not np.array_equal(got[:n], ref[p]):
            bad = np.nonzero(got[:n] != ref[p])[0]
            raise AssertionError(f"peer {p}: {bad.size} bytes differ, first at {bad[0]} "
                                 f"(row {bad[0] // rb}) W={W} rb={rb}")
        assert np.all(got[n:] == SENTINEL), f"peer {p}: bytes past the received rows written"
        assert outs[p].guards_intact(), f"peer {p}: canary before/after the output overwritten"
    for r in range(W):
        assert np.array_equal(ins[r].view.cpu().numpy(), inputs[r]), f"input {r} modified"
        assert ins[r].guards_intact(), f"input {r}: canary modified"
    return launch


def combine_checked(inputs, dispatch_so, rb, path=a2av.PATH_AUTO, in_mis=None, out_mis=None,
                    ctas_per_sm=0, expect_path=None):
    """Run the reverse exchange on the GPU and compare with the oracle's."""
    W = len(inputs)
    dso = np.ascontiguousarray(dispatch_so, dtype=np.int64).reshape(W, 2, W)
    in_mis = in_mis or [0] * W
    out_mis = out_mis or [0] * W
    back = [int(dso[:, 0, r].sum()) for r in range(W)]
    ins = [Guarded(inputs[p].size, in_mis[p], host=inputs[p]) for p in range(W)]
    outs = [Guarded((back[r] + SLACK_ROWS) * rb, out_mis[r], fill=SENTINEL) for r in range(W)]
    d_dso = torch.from_numpy(dso).cuda()
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    with a2av.A2av(W, path=path, ctas_per_sm=ctas_per_sm) as eng:
        eng.combine([g.view for g in ins], d_dso, [g.view for g in outs], so, rb)
        st = eng.status()
        launch = eng.last_launch()
    torch.cuda.synchronize()
    assert st == a2av.OK, f"device status {st}"
    if expect_path is not None:
        assert launch["path"] == expect_path, launch
    ref, ref_so = oracle.default().exchange_back(inputs, dso, rb)
    assert np.array_equal(so.cpu().numpy(), ref_so), "combine out_splits_offsets differ"
    for r in range(W):
        got = outs[r].view.cpu().numpy()
        n = back[r] * rb
        assert np.array_equal(got[:n], ref[r]), f"combine: rank {r} differs from the oracle"
        assert np.all(got[n:] == SENTINEL), f"combine: rank {r} written past its rows"
        assert outs[r].guards_intact(), f"combine: rank {r} canary overwritten"
    for p in range(W):
        assert np.array_equal(ins[p].view.cpu().numpy(), inputs[p]), f"combine input {p} modified"
    return [outs[r].view.cpu().numpy()[: back[r] * rb] for r in range(W)]


def dispatch_checked(K, rows, src, key, rb, rows_mis=None, out_mis=None, engine=None,
                     expect_copy=None, expect_kernels=None):
    """Fused dispatch on the GPU against the oracle's: outputs, offsets,
    positions and the split matrix; canaries and slack untouched.  With
    ``expect_copy`` / ``expect_kernels``, also that the library took that
    path (a2av_last_dispatch: the kernel that moved the rows, the number of
    kernels enqueued)."""
    W = len(rows)
    rows_mis = rows_mis or [0] * W
    out_mis = out_mis or [0] * W
    ref, ref_so, ref_pos, ref_S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    g_rows = [Guarded(rows[r].size, rows_mis[r], host=rows[r]) for r in range(W)]
    g_out = [Guarded(ref[p].size + SLACK_ROWS * rb, out_mis[p], fill=SENTINEL) for p in range(W)]
    d_src = [torch.from_numpy(np.ascontiguousarray(s, dtype=np.int32)).cuda() for s in src]
    d_key = [torch.from_numpy(np.ascontiguousarray(k, dtype=np.int32)).cuda() for k in key]
    d_pos = [torch.full((np.asarray(k).size,), -1, dtype=torch.int64, device="cuda") for k in key]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    isp = torch.full((W, W), -7, dtype=torch.int64, device="cuda")
    own = engine is None
    eng = engine or a2av.A2av(W)
    try:
        eng.dispatch([g.view for g in g_rows], d_src, d_key, K, [g.view for g in g_out], so, d_pos,
                     rb, in_splits=isp)
        st = eng.status()
        chain = eng.last_dispatch()
    finally:
        if own:
            eng.close()
    torch.cuda.synchronize()
    assert st == a2av.OK, f"device status {st}"
    assert np.array_equal(isp.cpu().numpy(), ref_S), "dispatch split matrix differs"
    assert np.array_equal(so.cpu().numpy(), ref_so), "dispatch out_splits_offsets differ"
    for r in range(W):
        assert np.array_equal(d_pos[r].cpu().numpy(), ref_pos[r]), f"rank {r}: positions differ"
    for p in range(W):
        got = g_out[p].view.cpu().numpy()
        n = ref[p].size
        if not np.array_equal(got[:n], ref[p]):
            bad = np.nonzero(got[:n] != ref[p])[0]
            raise AssertionError(f"dispatch peer {p}: {bad.size} bytes differ, first at row "
                                 f"{bad[0] // rb} (W={W} K={K} rb={rb})")
        assert np.all(got[n:] == SENTINEL), f"dispatch peer {p}: written past its rows"
        assert g_out[p].guards_intact(), f"dispatch peer {p}: canary overwritten"
    for r in range(W):
        assert np.array_equal(g_rows[r].view.cpu().numpy(), rows[r]), f"rows {r} modified"
    if expect_copy is not None:
        assert chain["copy_kernel"] == expect_copy, chain
    if expect_kernels is not None:
        assert chain["kernels"] == expect_kernels, chain
    return ref, ref_so, ref_pos, ref_S


def aligned_copy_kernel(rb: int, combine: bool = False) -> str:
    """The kernel that moves 16-byte aligned rows of rb bytes past the
    one-kernel size: the cp.async.bulk gather for rows above 2 KiB .. 32 KiB
    (the combine: from 64 B), register copies otherwise."""
    lo = 64 if combine else 2049
    return "dispatch_gather_kernel" if lo <= rb <= 32768 else "dispatch_copy_kernel"
