"""One small pass of the whole hot path on cuda:0, checked against the CPU oracle.

Used by ``__graft_entry__.smoke()``; it lives with the tests because it
calls the CPU oracle, which the library package never imports.  Workload:
the toy shape (batch 1, d 256, 4/2 heads x 64, V 1024, ctx 128, depth 4,
top-k 4, budget 16), fp32:
  draft round : LM-head top-k on synthetic drafter rows + tree expansion per
                depth, then rerank/flatten
  drafter     : the input FC with the embedding lookup and the decoder layer
                over the frontier rows (fp32 and bf16)
  verify      : tree attention, fused projection, LM head (k = 1), greedy
                and stochastic verification, and stochastic verification from
                LM-head statistics
"""
import numpy as np
import torch


def run(device="cuda:0"):
    import oracle  # test infrastructure: the checker of the smoke pass
    from eagle_speculative_decoding_gb300 import binding as b
    from eagle_speculative_decoding_gb300 import synth

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

    # drafter decoder layer over the frontier rows (rows 1..width of its tree,
    # each below row 0), fp32 and bf16
    Hq_, Hkv_, D_, I_ = c["Hq"], c["Hkv"], c["D"], synth.FFN_WIDTH[d]
    Rm, r0 = 1 + width, 1
    wl = dict(norm1=1 + 0.1 * synth.normal((d,), 1.0, dt, gen),
              qkv=synth.normal(((Hq_ + 2 * Hkv_) * D_, d), 0.05, dt, gen),
              o=synth.normal((d, Hq_ * D_), 0.05, dt, gen),
              norm2=1 + 0.1 * synth.normal((d,), 1.0, dt, gen),
              gu=synth.normal((2 * I_, d), 0.05, dt, gen), down=synth.normal((d, I_), 0.05, dt, gen))
    par = np.array([-1] + [0] * width)
    lmask = oracle.ancestor_mask(par)[None]
    lpos = (ctx.numpy()[:, None] + 1).repeat(width, axis=1).astype(np.int32)
    for ddt, tol in ((torch.float32, 1e-4), (torch.bfloat16, 2e-2)):
        xin = g[: B * width].to(ddt)
        kt0 = synth.normal((B, Rm, Hkv_, D_), 1.0, ddt, gen)
        vt0 = synth.normal((B, Rm, Hkv_, D_), 1.0, ddt, gen)
        qt_d = torch.zeros((B, Rm, Hq_, D_), dtype=ddt, device=dev)
        kt_d, vt_d = kt0.to(dev), vt0.to(dev)
        lo = torch.empty_like(xin)
        b.eagle_draft_layer(xin, {k_: v_.to(dev, ddt) for k_, v_ in wl.items()}, torch.from_numpy(lpos).to(dev),
                            kc.to(dev, ddt), vc.to(dev, ddt), table.to(dev), ctx.to(dev), qt_d, kt_d, vt_d,
                            torch.from_numpy(lmask.view(np.int64)).to(dev), r0, lo, status=status)
        store = None if ddt == torch.float32 else (
            lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy())
        f64 = lambda t: t.to(ddt).double().cpu().numpy()
        ref_l, _, _ = oracle.draft_layer(f64(xin), {k_: f64(v_) for k_, v_ in wl.items()}, lpos, f64(kc), f64(vc),
                                         table.numpy(), ctx.numpy(), f64(kt0), f64(vt0), lmask, r0, Hq_, Hkv_,
                                         store=store)
        err = np.abs(lo.double().cpu().numpy() - ref_l).max() / (np.abs(ref_l).max() + 1e-30)
        assert err < tol, ("draft_layer", ddt, err)

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
