"""Helpers of the GPU tests: run the library's stages through the C-ABI binding and read
back the workspace regions, and compare against the oracle."""
import numpy as np
import torch

TOL = {"a16w16": 2e-2, "a8w8_int8": 2e-2, "a8w4_int": 2e-2, "a8w8_fp8": 6e-2, "a8w4_fp8_fp4": 6e-2,
       "a8w8_fp8_e5m2": 6e-2}


def lib():
    import __graft_entry__
    __graft_entry__.build_module().build()
    import moe_expert_ffn_topk_gb300 as moe
    return moe


def run_forward(moe, wl, inp, flags=0, stages=False, shared=0):
    """One forward pass; returns y (and, with stages=True, the plan and workspace views).
    With shared > 0 the weights hold wl.E routed experts followed by the shared ones."""
    dev = inp["topk_ids"].device
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K, shared)
    ws = moe.alloc_workspace(d, wl.mode, dev)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=dev)
    if stages:
        E, K = wl.E + shared, wl.K + shared  # the plan covers the shared experts' slots too
        counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
        offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
        row_src = torch.full((max(wl.T * K, 1),), -7, dtype=torch.int32, device=dev)
        moe.moe_plan(inp["topk_ids"], d, ws, counts, offsets, row_src)
        moe.moe_dispatch(inp["x"], inp["x_scale"], d, wl.mode, ws)
        moe.moe_expert_l1(inp["w1"], inp["w1_scale"], d, wl.mode, ws, flags)
        moe.moe_expert_l2(inp["w2"], inp["w2_scale"], inp["topk_weights"], d, wl.mode, ws, flags)
        moe.moe_combine(y, d, ws)
    else:
        moe.moe_forward(inp["x"], inp["x_scale"], inp["topk_ids"], inp["topk_weights"], inp["w1"], inp["w1_scale"],
                        inp["w2"], inp["w2_scale"], y, d, wl.mode, ws, flags)
    status = moe.moe_check_device_error(ws)
    out = {"y": y, "status": status, "ws": ws, "d": d}
    if stages:
        L = moe.moe_workspace_layout(d, wl.mode)
        out.update(counts=counts, offsets=offsets, row_src=row_src[:wl.T * (wl.K + shared)], layout=L)
    return out


def region(ws, L, name, dtype, count):
    off = L[name]
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def y_numpy(y):
    return y.float().cpu().double().numpy()


def assert_close(got, ref, mode, what="y"):
    err = np.abs(got - ref).max() if got.size else 0.0
    bound = TOL[mode] * (np.abs(ref).max() if ref.size else 0.0)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= bound, f"{what}: max|got - ref| = {err:.4e} > {bound:.4e} ({TOL[mode]} * max|ref|)"
    return err, bound


def slice_tokens(inp, tokens):
    """The inputs of a subset of tokens (tokens are independent problems)."""
    idx = torch.as_tensor(tokens, device=inp["topk_ids"].device, dtype=torch.long)
    out = dict(inp)
    for k in ("x", "topk_ids", "topk_weights"):
        out[k] = inp[k].index_select(0, idx).contiguous()
    if inp["x_scale"] is not None:
        out["x_scale"] = inp["x_scale"].index_select(0, idx).contiguous()
    return out


def covering_tokens(topk_ids, seed, extra=2):
    """A sample of tokens in which every expert that any token routes to appears at least once
    (greedy set cover in a seeded order), plus `extra` more seeded tokens. Sorted token indices."""
    ids = np.asarray(topk_ids)
    rng = np.random.default_rng(seed)
    sets = [set(int(e) for e in row if e >= 0) for row in ids]
    uncovered = set().union(*sets) if sets else set()
    order = [int(t) for t in rng.permutation(ids.shape[0])]
    chosen = []
    while uncovered:
        best = max(order, key=lambda t: len(sets[t] & uncovered))
        chosen.append(best)
        uncovered -= sets[best]
    chosen += [t for t in order if t not in chosen][:extra]
    return sorted(chosen)


def _oracle_chunk(args):
    from oracle import moe as omoe
    mode, h, inter, clamp = args
    return omoe.forward(mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                        h["w2"], h["w2_scale"], num_experts=h["w1"].shape[0], inter=inter, clamp=clamp)


def oracle_tokens(mode, h, tokens, inter, workers=8, clamp=None):
    """The oracle's y for a subset of tokens of host inputs h (numpy), computed in `workers` spawned
    processes: every token is an independent problem and every expert an independent FFN, so each
    chunk of tokens runs the oracle on the experts it routes to only (their weights sliced out, ids
    renumbered). Returns y rows in the order of `tokens`."""
    import concurrent.futures
    import multiprocessing
    tokens = list(tokens)
    chunks = [tokens[i::workers] for i in range(min(workers, len(tokens)))]
    jobs = []
    for ch in chunks:
        ids = h["topk_ids"][ch]
        used = np.unique(ids[ids >= 0])
        local = np.full(int(used.max()) + 1 if used.size else 1, -1, np.int64)
        local[used] = np.arange(used.size)
        sub = {"x": h["x"][ch], "x_scale": None if h["x_scale"] is None else h["x_scale"][ch],
               "topk_ids": np.where(ids >= 0, local[np.maximum(ids, 0)], -1).astype(np.int32),
               "topk_weights": h["topk_weights"][ch]}
        for k in ("w1", "w1_scale", "w2", "w2_scale"):
            sub[k] = None if h[k] is None else np.ascontiguousarray(h[k][used])
        jobs.append((mode, sub, inter, clamp))
    ctx = multiprocessing.get_context("spawn")  # never fork a process that holds a CUDA context
    with concurrent.futures.ProcessPoolExecutor(max_workers=len(jobs), mp_context=ctx) as ex:
        outs = list(ex.map(_oracle_chunk, jobs))
    y = np.zeros((len(tokens), outs[0].shape[1]))
    pos = {t: i for i, t in enumerate(tokens)}
    for ch, out in zip(chunks, outs):
        for j, t in enumerate(ch):
            y[pos[t]] = out[j]
    return y
