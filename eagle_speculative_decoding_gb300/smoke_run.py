"""One small pass of the whole hot path on cuda:0, checked against the CPU oracle.

Used by ``__graft_entry__.smoke()``.  Workload: the toy shape (batch 1,
d 256, 4/2 heads x 64, V 1024, ctx 128, depth 4, top-k 4, budget 16), fp32:
  draft round : LM-head top-k on synthetic drafter rows + tree expansion per
                depth, then rerank/flatten
  verify      : tree attention, fused projection, LM head (k = 1), greedy
                and stochastic verification, and stochastic verification from
                LM-head statistics
"""
import numpy as np
import torch


def run(device="cuda:0"):
    import oracle  # test infrastructure, allowed here
    from . import binding as b
    from . import synth

    torch.cuda.set_device(device)
    c = synth.CONFIGS["toy"]
    B, d, V, k, width, depth, N = c["B"], c["d"], c["V"], c["topk"], c["width"], c["depth"], c["N"]
    R = N + 1
    dt = torch.float32
    gen = synth.generator(0)
    dev = device
    w_lm = synth.normal((V, d), synth.WEIGHT_STD, dt, gen)
    w_proj = synth.normal((d, 3 * d), synth.WEIGHT_STD, dt, gen)
    root = synth.random_tokens((B,), V, gen)
    max_nodes = 1 + synth.n_candidates(c)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # ---- draft round
    st_ref = oracle.tree_expand_init(int(root[0]))
    z32 = lambda *s, t=torch.int32: torch.zeros(s, dtype=t, device=dev)
    parent, token, logv, ndepth = z32(B, max_nodes), z32(B, max_nodes), z32(B, max_nodes, t=torch.float32), z32(B, max_nodes)
    count, frontier, nf = z32(B), z32(B, width), z32(B)
    w_lm_d = w_lm.to(dev)
    for s in range(depth):
        P = 1 if s == 0 else width
        x = synth.normal((B * P, d), 1.0, dt, gen)
        ids = torch.empty((B * P, k), dtype=torch.int32, device=dev)
        lps = torch.empty((B * P, k), dtype=torch.float32, device=dev)
        b.eagle_lmhead_topk(x.to(dev), w_lm_d, k, ids, lps, status=status)
        ref = oracle.lmhead_topk(x.numpy(), w_lm.numpy(), k)
        g_ids = ids.cpu().numpy()
        npar = len(st_ref["frontier"])
        assert np.array_equal(g_ids[:npar], ref["ids"][:npar]), "lmhead top-k ids"
        assert np.abs(lps.cpu().numpy()[:npar] - ref["logprobs"][:npar]).max() < 1e-3
        b.eagle_tree_expand(s, width, ids.view(B, P, k), lps.view(B, P, k), root.to(dev), parent,
                            token, logv, ndepth, count, frontier, nf, status=status)
        oracle.tree_expand_step(st_ref, g_ids[:npar], lps.cpu().numpy()[:npar], width)
    ctx = synth.ctx_lengths(c, gen)
    flat = {n: z32(B, R) for n in ("token", "parent_row", "depth", "node_id", "position")}
    flat["mask"] = z32(B, R, t=torch.int64)
    flat["n_rows"] = z32(B)
    b.eagle_tree_expand_finalize(N, parent, token, logv, ndepth, count, ctx.to(dev), flat["token"],
                                 flat["parent_row"], flat["depth"], flat["mask"], flat["node_id"],
                                 flat["position"], flat["n_rows"], status=status)
    ref_flat = oracle.tree_expand_finalize(st_ref, N, int(ctx[0]), R_out=R)
    for key in ("token", "parent_row", "node_id", "position"):
        assert np.array_equal(flat[key].cpu().numpy()[0], ref_flat[key]), key

    # ---- verify
    Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
    q = synth.normal((B, R, Hq, D), 1.0, dt, gen)
    kt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    vt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    kc, vc, table = synth.paged_kv(ctx.tolist(), Hkv, D, 16, dt, gen)
    out = torch.empty((B, R, Hq, D), dtype=dt, device=dev)
    b.eagle_tree_attn(q.to(dev), kt.to(dev), vt.to(dev), kc.to(dev), vc.to(dev), table.to(dev),
                      ctx.to(dev), flat["mask"], out, status=status)
    ref_o, _ = oracle.tree_attn(q.numpy(), kt.numpy(), vt.numpy(), kc.numpy(), vc.numpy(),
                                table.numpy(), ctx.numpy(), ref_flat["mask"][None])
    assert np.abs(out.cpu().numpy() - ref_o).max() < 1e-3, "tree attention"

    hs = [synth.normal((B * R, d), 1.0, dt, gen) for _ in range(3)]
    g = torch.empty((B * R, d), dtype=dt, device=dev)
    b.eagle_fuse_proj(*(h.to(dev) for h in hs), w_proj.to(dev), g, status=status)
    ref_g = oracle.fuse_proj(*(h.numpy() for h in hs), w_proj.numpy())
    assert np.abs(g.cpu().numpy() - ref_g).max() < 1e-2 * (np.abs(ref_g).max() + 1), "fuse_proj"

    # drafter input FC over the frontier rows, fp32 and bf16 (tensor cores)
    w_in = synth.normal((d, 2 * d), synth.WEIGHT_STD, dt, gen)
    toks = synth.random_tokens((B * width,), V, gen)
    for ddt, tol in ((torch.float32, 1e-4), (torch.bfloat16, 2e-2)):
        r_in = g[: B * width].to(ddt)
        u = torch.empty((B * width, d), dtype=ddt, device=dev)
        b.eagle_draft_input(r_in, toks.to(dev), w_lm.to(dev, ddt), w_in.to(dev, ddt), u, status=status)
        ref_u = oracle.draft_input(r_in.float().cpu().numpy(), toks.numpy(), w_lm.to(ddt).float().numpy(),
                                   w_in.to(ddt).float().numpy())
        err = np.abs(u.float().cpu().numpy() - ref_u).max() / (np.abs(ref_u).max() + 1e-30)
        assert err < tol, ("draft_input", ddt, err)

    am = torch.empty((B * R, 1), dtype=torch.int32, device=dev)
    amlp = torch.empty((B * R, 1), dtype=torch.float32, device=dev)
    b.eagle_lmhead_topk(g, w_lm_d, 1, am, amlp, status=status)
    acc = z32(B)
    path = z32(B, depth + 1)
    toks = z32(B, depth + 1)
    b.eagle_tree_verify(flat["parent_row"], flat["token"], 0.0, depth, acc, path, toks,
                        n_rows=flat["n_rows"], target_argmax=am.view(B, R), V=V, status=status)
    ref_v = oracle.tree_verify(ref_flat["parent_row"][None], ref_flat["token"][None], 0.0, depth,
                               n_rows=[ref_flat["n_rows"]], target_argmax=am.view(B, R).cpu().numpy())
    assert np.array_equal(toks.cpu().numpy(), ref_v["out_tokens"]), "greedy verify"

    logits = synth.target_logits((B, R, V), gen)
    b.eagle_tree_verify(flat["parent_row"], flat["token"], 1.0, depth, acc, path, toks,
                        n_rows=flat["n_rows"], target_logits=logits.to(dev), seed=7, status=status)
    ref_s = oracle.tree_verify(ref_flat["parent_row"][None], ref_flat["token"][None], 1.0, depth,
                               n_rows=[ref_flat["n_rows"]], target_logits=logits.numpy(), seed=7)
    if min((m for _, _, m in ref_s["margins"]), default=1.0) > 1e-5:
        assert np.array_equal(toks.cpu().numpy(), ref_s["out_tokens"]), "stochastic verify"
    # stochastic verification from LM-head statistics (no [B, R, V] logits)
    rk = k + 1
    xv = synth.normal((B * R, d), 1.0, dt, gen)
    st_out = dict(ids=z32(B * R, rk), keys=z32(B * R, rk, t=torch.float32),
                  m=z32(B * R, t=torch.float32), s=z32(B * R, t=torch.float32),
                  c=z32(B * R, t=torch.float32))
    b.eagle_lmhead_verify_stats(xv.to(dev), w_lm_d, flat["parent_row"], flat["token"], 1.0, rk,
                                st_out["ids"], st_out["keys"], st_out["m"], st_out["s"],
                                st_out["c"], n_rows=flat["n_rows"], seed=9, status=status)
    b.eagle_tree_verify_stats(flat["parent_row"], flat["token"], 1.0, depth, st_out["m"],
                              st_out["s"], st_out["c"], st_out["ids"], acc, path, toks, V,
                              n_rows=flat["n_rows"], seed=9, status=status)
    ref_st = oracle.verify_stats(xv.numpy(), w_lm.numpy(), ref_flat["parent_row"][None],
                                 ref_flat["token"][None], 1.0, rk, seed=9, n_rows=[ref_flat["n_rows"]])
    assert np.abs(st_out["m"].cpu().numpy() - ref_st["row_max"]).max() < 1e-3, "row max"
    ref_w = oracle.tree_verify(ref_flat["parent_row"][None], ref_flat["token"][None], 1.0, depth,
                               n_rows=[ref_flat["n_rows"]],
                               target_logits=(xv.double() @ w_lm.double().T).reshape(B, R, V).numpy(),
                               seed=9)
    if min((m for _, _, m in ref_w["margins"]), default=1.0) > 1e-4:
        assert np.array_equal(toks.cpu().numpy(), ref_w["out_tokens"]), "verify from statistics"
    torch.cuda.synchronize()
    assert int(status.item()) == 0, b.STATUS.get(int(status.item()))
    print("smoke ok: launches", b.launch_count())
