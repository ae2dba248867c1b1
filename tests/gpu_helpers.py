"""Shared helpers for the GPU parity tests: tolerances and oracle-on-slices."""
import numpy as np
import torch

import oracle

# Tolerances stated for this operation: bf16 inputs with fp32 accumulation to
# max-abs <= 2e-2 and mean-abs <= 2e-3 on the output; LSE to 1e-3 absolute;
# fp32 paths to 1e-5 relative (read normwise: max|err| / max|ref|).
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
F32_REL = 1e-5


def assert_bf16_close(got, ref, what="out"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    assert err.max() <= BF16_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"


def assert_lse_close(got, ref, tol=LSE_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), "lse: non-finite values"
    err = np.abs(got - ref).max()
    assert err <= tol, f"lse: max abs err {err:.3e}"


def assert_f32_close(got, ref, what="out", tol=F32_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert rel <= tol, f"{what}: normwise rel err {rel:.3e}"


def oracle_rows_from_slices(q, k, v, sink, W, rows):
    """Oracle values for selected rows (b, h, i) of a large problem.

    Each row depends only on keys/values in [max(0, i-W+1), i] of its batch
    entry, so the oracle runs on that slice alone (copied to the host), which
    gives exactly the same result as running it on the whole input.
    Returns (out [n, D], lse [n]) in fp64, in the order of ``rows``.
    """
    n = len(rows)
    D = q.shape[-1]
    out = np.zeros((n, D))
    lse = np.zeros(n)
    groups = {}
    for idx, (b, h, i) in enumerate(rows):
        groups.setdefault((int(b), int(i)), []).append((idx, int(h)))
    sink_c = sink.detach().cpu()
    for (b, i), members in groups.items():
        j0 = max(0, i - W + 1)
        L = i - j0 + 1
        # the oracle reads only query row i: leave the other rows zero
        qs = torch.zeros((1, L) + tuple(q.shape[2:]), dtype=q.dtype)
        qs[0, L - 1] = q[b, i].cpu()
        ks = k[b:b + 1, j0:i + 1].cpu()
        vs = v[b:b + 1, j0:i + 1].cpu()
        sel = [[0, h, L - 1] for _, h in members]
        o, l = oracle.swa_sink_fwd_rows(qs, ks, vs, sink_c, W, sel)
        for m, (idx, _) in enumerate(members):
            out[idx] = o[m]
            lse[idx] = l[m]
    return out, lse


def oracle_by_slices(q, k, v, sink, W, b, s0, s1):
    """Oracle values of positions s0..s1-1 of batch entry b, every head:
    (out [s1-s0, Hq, D], lse [Hq, s1-s0]) in fp64.

    The oracle runs on positions max(0, s0-W+1) .. s1-1 only.  A row i >= s0
    reads keys [max(0, i-W+1), i], all inside that range, so its value is the
    one the oracle gives on the whole sequence; the W-1 halo rows before s0
    are computed with truncated windows and dropped."""
    j0 = max(0, s0 - W + 1)
    qs, ks, vs = (t[b:b + 1, j0:s1].cpu() for t in (q, k, v))
    o, l = oracle.swa_sink_fwd(qs, ks, vs, sink.detach().cpu(), W)
    return o[0, s0 - j0:], l[0, :, s0 - j0:]


def gather_rows(out, lse, rows):
    """Kernel outputs at the selected rows, as fp64 numpy arrays."""
    idx_b = torch.tensor([r[0] for r in rows])
    idx_h = torch.tensor([r[1] for r in rows])
    idx_i = torch.tensor([r[2] for r in rows])
    o = out[idx_b.to(out.device), idx_i.to(out.device), idx_h.to(out.device)]
    l = lse[idx_b.to(lse.device), idx_h.to(lse.device), idx_i.to(lse.device)]
    return o.double().cpu().numpy(), l.double().cpu().numpy()


def sample_rows(B, T, Hq, n_pos, seed, extra_pos=(), heads=None):
    """Deterministic sample of (b, h, i): chosen positions with all (or given) heads."""
    g = np.random.default_rng(seed)
    pos = set(int(p) for p in extra_pos if 0 <= p < T)
    pos |= {0, 1, 15, 16, 127, 128, 129, T - 1, T - 2, T - 17}
    pos = {p for p in pos if 0 <= p < T}
    while len(pos) < n_pos and len(pos) < T:
        pos.add(int(g.integers(0, T)))
    hs = list(range(Hq)) if heads is None else list(heads)
    rows = []
    for i in sorted(pos):
        b = int(g.integers(0, B))
        for h in hs:
            rows.append((b, h, i))
    return rows


def oracle_block_scores_from_slices(q, k, entries):
    """Oracle block scores of the global layer (every causal pair, W >= T) at
    selected entries (b, g, kb): query group g (positions 4g..4g+3), key block
    kb (keys 128kb..128kb+127).  Returns [n, Hkv] fp64.

    An entry depends only on those 4 query rows, those 128 key rows and on
    which pairs satisfy j <= i.  Shifting every position by -128kb keeps the
    block at keys 0..127.  A group that overlaps the block keeps its offset
    (at most 124); a group past the block goes to sub-positions 128..131,
    where it sees every key of the block, as it does in the whole sequence.
    The oracle then runs on that short sequence alone.
    """
    out = []
    for b, g, kb in entries:
        p0, j0 = 4 * int(g), 128 * int(kb)
        assert j0 <= p0 + 3, "block after the query group: no valid pair"
        off = p0 - j0 if p0 - j0 < 128 else 128
        L = off + 4
        n = min(128, L)
        qs = torch.zeros((1, L) + tuple(q.shape[2:]), dtype=q.dtype)
        ks = torch.zeros((1, L) + tuple(k.shape[2:]), dtype=k.dtype)
        qs[0, off:off + 4] = q[int(b), p0:p0 + 4].cpu()
        ks[0, :n] = k[int(b), j0:j0 + n].cpu()
        out.append(oracle.block_max(qs, ks, L)[0, :, off // 4, 0])
    return np.array(out)


def oracle_sparse_rows_from_slices(q, k, v, sink, idx, QB, rows):
    """Oracle outputs of the sparse layer at selected rows (b, h, i), for the
    block selection idx [B, Hkv, ceil(T/QB), topk] (-1 = none).

    Row i of head h attends to the keys j <= i of the blocks selected for its
    query block and its kv head, with the sink.  Those keys, gathered in
    increasing order into a short sequence, followed by the query at the last
    of its sub-positions, give a causal row that sees exactly them, so the
    prefill oracle's row is the sparse layer's row.
    Returns (out [n, D], lse [n]) fp64.
    """
    Hq, D = q.shape[2], q.shape[3]
    Hkv = k.shape[2]
    G = Hq // Hkv
    idx = np.asarray(idx.cpu() if isinstance(idx, torch.Tensor) else idx)
    sink_c = sink.detach().cpu()
    out = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    for r, (b, h, i) in enumerate(rows):
        b, h, i = int(b), int(h), int(i)
        kvh = h // G
        sel = [int(kb) for kb in idx[b, kvh, i // QB] if kb >= 0 and 128 * kb <= i]
        if not sel:
            out[r] = 0.0
            lse[r] = float(sink_c[h])
            continue
        J = torch.from_numpy(np.concatenate(
            [np.arange(128 * kb, min(128 * kb + 128, i + 1)) for kb in sel]))
        n = len(J)
        qs = torch.zeros((1, n, G, D), dtype=q.dtype)
        qs[0, n - 1] = q[b, i, kvh * G:(kvh + 1) * G].cpu()
        ks = k[b, :, kvh:kvh + 1].cpu()[J].unsqueeze(0)
        vs = v[b, :, kvh:kvh + 1].cpu()[J].unsqueeze(0)
        o, l = oracle.swa_sink_fwd_rows(qs, ks, vs, sink_c[kvh * G:(kvh + 1) * G], n,
                                        [[0, h - kvh * G, n - 1]])
        out[r] = o[0]
        lse[r] = l[0]
    return out, lse
