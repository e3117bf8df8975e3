"""A check of a top-K cache (ids, logp) against the logits x it came from, by
properties that hold at any size and together fix the answer exactly:

  * ids in [0, V); values non-increasing, and ascending ids where values are
    equal (so the ids are distinct);
  * every element above the K-th chosen value is chosen;
  * the chosen elements equal to the K-th value are the lowest ids with that
    value (ties to the lowest id; -0.0 equals +0.0);
  * logp = x[id] - logsumexp(x) (fp64) within `tol`.

It runs in blocks of rows with torch on whatever device x is on."""

import torch


def check_topk_rows(x: torch.Tensor, ids: torch.Tensor, logp: torch.Tensor, tol: float, block: int = 1024):
    R, V = x.shape
    K = ids.shape[1]
    for r0 in range(0, R, block):
        xf = x[r0:r0 + block].float()
        ic = ids[r0:r0 + block].long()
        lp = logp[r0:r0 + block].double()
        assert int(ic.min()) >= 0 and int(ic.max()) < V, "id out of range"
        vals = torch.gather(xf, 1, ic)
        assert bool((vals[:, 1:] <= vals[:, :-1]).all()), "values increase"
        eq = vals[:, 1:] == vals[:, :-1]
        assert bool((ic[:, 1:][eq] > ic[:, :-1][eq]).all()), "equal values not in ascending id order"
        vK = vals[:, K - 1:K]
        n_gt_sel = (vals > vK).sum(1)
        assert torch.equal((xf > vK).sum(1), n_gt_sel), "an element above the K-th value is missing"
        m = (K - n_gt_sel)[:, None]
        rank = (xf == vK).to(torch.int32).cumsum(1)  # 1-based rank by id among elements equal to vK
        r_sel = torch.gather(rank, 1, ic)
        at_k = vals == vK
        assert bool((r_sel <= m)[at_k].all()), "a tie at the K-th value did not go to the lowest id"
        lse = torch.logsumexp(xf.double(), dim=1, keepdim=True)
        err = (lp - (vals.double() - lse)).abs().max().item()
        assert err <= tol, "logp off by %g" % err
