"""Helpers shared by the GPU parity tests: seeded inputs on both sides, the
output tolerance, and the mapping between the GPU's padded sorted rows and
the oracle's unpadded ones."""
import numpy as np
import torch

import moe_inputs as mi
import oracle
import block_fp8_mixture_topk_gb300 as moe

# Output tolerance of the layer: relative Frobenius error and per-element error
# against the root-mean-square of the reference.
REL_FRO = 1e-2
MAX_REL_RMS = 5e-2


def assert_output_close(got_bf16: torch.Tensor, ref: np.ndarray, rows=None):
    got = got_bf16.float().cpu().double().numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.all(np.isfinite(got)), "non-finite output"
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2))
    worst = np.abs(got - ref).max() / rms
    assert rel <= REL_FRO and worst <= MAX_REL_RMS, f"rel_fro={rel:.3e} max|d|/rms={worst:.3e}"
    return rel, worst


def routing_of(wl: mi.Workload, device="cuda"):
    bias = mi.expert_bias(wl)
    if wl.scoring == mi.SIGMOID:
        rp = moe.RoutingParams("sigmoid", wl.n_group, wl.topk_group, wl.routed_scaling,
                               None if bias is None else bias.to(device))
    else:
        rp = moe.RoutingParams("softmax", 1, 1, wl.routed_scaling)
    okw = dict(scoring=wl.scoring, bias=None if bias is None else bias.numpy(), n_group=wl.n_group,
               topk_group=wl.topk_group, routed_scaling=wl.routed_scaling)
    return rp, okw


class Layer:
    """Quantised weights of a workload on the GPU (GPU quantiser), plus the
    oracle's own quantisation of any subset of experts (from the same bf16)."""

    def __init__(self, wl: mi.Workload, device="cuda", chunk=8, scale_fmt="f32"):
        self.wl, self.device, self.scale_fmt = wl, device, scale_fmt
        E, H, I = wl.E, wl.H, wl.I
        self.w13q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
        self.w13s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=device)
        self.w2q = torch.empty(E, H, I, dtype=torch.uint8, device=device)
        self.w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=device)
        for e0 in range(0, E, chunk):
            ex = range(e0, min(E, e0 + chunk))
            q, s = moe.fp8_block_quant_weight(mi.w13_bf16(wl, device, ex), scale_fmt)
            self.w13q[e0:e0 + len(ex)], self.w13s[e0:e0 + len(ex)] = q, s
            q, s = moe.fp8_block_quant_weight(mi.w2_bf16(wl, device, ex), scale_fmt)
            self.w2q[e0:e0 + len(ex)], self.w2s[e0:e0 + len(ex)] = q, s
        torch.cuda.synchronize()

    def oracle_weights(self, experts):
        """Oracle-quantised weights as full [E, ...] arrays with only `experts` filled."""
        wl = self.wl
        experts = sorted(set(int(e) for e in experts))
        E, H, I = wl.E, wl.H, wl.I
        w13q = np.zeros((E, 2 * I, H), dtype=np.uint8)
        w13s = np.zeros((E, 2 * I // 128, H // 128), dtype=np.float32)
        w2q = np.zeros((E, H, I), dtype=np.uint8)
        w2s = np.zeros((E, H // 128, I // 128), dtype=np.float32)
        fmt = oracle.SCALE_UE8M0 if self.scale_fmt == "ue8m0" else oracle.SCALE_F32
        for e in experts:
            w13q[e], w13s[e] = [a[0] for a in oracle.quant_128x128_bf16(
                mi.bf16_bits(mi.w13_bf16(wl, self.device, [e])), fmt)]
            w2q[e], w2s[e] = [a[0] for a in oracle.quant_128x128_bf16(
                mi.bf16_bits(mi.w2_bf16(wl, self.device, [e])), fmt)]
        return w13q, w13s, w2q, w2s

    def forward(self, hidden, logits, rp, packed=False):
        w13, w2 = self.w13q, self.w2q
        if packed:
            w13, w2 = moe.moe_fp8_block_pack_weights(w13), moe.moe_fp8_block_pack_weights(w2)
        return moe.moe_fp8_block_forward(hidden, logits, w13, self.w13s, w2, self.w2s, self.wl.topk,
                                         self.wl.renormalize, rp, scale_fmt=self.scale_fmt)


def unpadded_rows(padded_offsets: np.ndarray, offsets: np.ndarray):
    """Index array mapping the oracle's sorted row i to the GPU's padded row."""
    E = offsets.size - 1
    out = np.empty(offsets[-1], dtype=np.int64)
    for e in range(E):
        n = offsets[e + 1] - offsets[e]
        out[offsets[e]:offsets[e + 1]] = padded_offsets[e] + np.arange(n)
    return out


def check_sort(perm, ids_np, E, block_m=128):
    """The GPU's expert sort (outputs of moe_align_permute or its no-workspace variant) against
    the oracle's stable sort of the same ids, bit for bit: offsets, padded offsets, the pair of
    every real row, -1 in every padding row, the unpermute map and the tile table."""
    off, sorted_, pos = oracle.permute(ids_np, E)
    counts = np.diff(off)
    padded = (counts + block_m - 1) // block_m * block_m
    poff = np.concatenate([[0], np.cumsum(padded)])
    assert np.array_equal(perm["expert_offsets"].cpu().numpy(), off)
    assert np.array_equal(perm["padded_offsets"].cpu().numpy(), poff)
    rows = unpadded_rows(poff, off)
    sp = perm["sorted_pair_ids"].cpu().numpy()
    assert np.array_equal(sp[rows], sorted_)
    pad = np.ones(poff[-1], dtype=bool)
    pad[rows] = False
    assert np.all(sp[:poff[-1]][pad] == -1)
    assert np.array_equal(perm["pos"].cpu().numpy()[:ids_np.size], rows[pos])
    nt = int(perm["num_tiles"].item())
    assert nt == poff[-1] // block_m
    te = perm["tile_expert"].cpu().numpy()[:nt]
    tr = perm["tile_row0"].cpu().numpy()[:nt]
    assert np.array_equal(tr, np.arange(nt) * block_m)
    assert np.array_equal(te, np.searchsorted(poff, tr, side="right") - 1)


def tile_sample_tokens(oids: np.ndarray, E: int, block_m: int = 128, extra=()):
    """Tokens that cover every expert tile of a routed step: for each padded tile of
    block_m rows, the token owning its last real row, and for each expert the token owning its
    first row (rows in the sort's order: by expert, pairs p = t*topk + j ascending).  `extra`
    tokens are added.  Returns a sorted list."""
    topk = oids.shape[1]
    off, sorted_, _ = oracle.permute(oids, E)
    toks = set(int(t) for t in extra)
    for e in range(E):
        n = int(off[e + 1] - off[e])
        if n == 0:
            continue
        toks.add(int(sorted_[off[e]]) // topk)
        for last in range(block_m - 1, n + block_m - 1, block_m):
            toks.add(int(sorted_[off[e] + min(last, n - 1)]) // topk)
    return sorted(toks)
