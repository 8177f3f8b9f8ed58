"""Helpers for the GPU parity tests: tolerance checks and small batch builders."""
from __future__ import annotations

import numpy as np
import torch

# Tolerance for bf16 inputs with fp32 accumulation (and the fp32 path), against
# the float64 oracle: max-abs error and relative RMS error.
MAX_ABS = 2e-2
REL_RMS = 5e-3
LSE_ABS = 2e-3


def check_close(got: torch.Tensor, ref: np.ndarray, what: str = "", max_abs=MAX_ABS, rel_rms=REL_RMS):
    g = got.detach().double().cpu().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    rr = float(np.sqrt((err ** 2).sum() / max((ref ** 2).sum(), 1e-300)))
    ma = float(err.max()) if err.size else 0.0
    assert ma <= max_abs and rr <= rel_rms, f"{what}: max-abs {ma:.3e} (<= {max_abs}), rel-RMS {rr:.3e} (<= {rel_rms})"
    return ma, rr


def i32(x, device="cuda"):
    return torch.tensor(list(x), dtype=torch.int32, device=device)


def varlen_batch(seed, lens, h_q, h_kv, d, dtype=torch.bfloat16, device="cuda", std=0.5, spare_pages=3):
    """Random varlen batch (P_s, E_s) with shuffled pages; every cache page is
    filled (so slots past a sequence's end hold finite values), the new rows
    are separate tensors to append."""
    g = torch.Generator().manual_seed(seed)
    pg = 16
    npages = [max(1, -(-(P + E) // pg)) for P, E in lens]
    total = sum(npages) + spare_pages
    order = torch.randperm(total, generator=g)
    max_pages = max(npages)
    pt = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(npages):
        pt[s, :n] = order[off:off + n].to(torch.int32)
        off += n
    kc = (torch.randn(total, pg, h_kv, d, generator=g) * std).to(dtype)
    vc = (torch.randn(total, pg, h_kv, d, generator=g) * std).to(dtype)
    total_q = sum(E for _, E in lens)
    q = (torch.randn(total_q, h_q, d, generator=g) * std).to(dtype)
    kn = (torch.randn(total_q, h_kv, d, generator=g) * std).to(dtype)
    vn = (torch.randn(total_q, h_kv, d, generator=g) * std).to(dtype)
    qo = [0]
    for _, E in lens:
        qo.append(qo[-1] + E)
    pl = [P for P, _ in lens]
    max_kv = max(P + E for P, E in lens)
    return dict(q=q.to(device), k_new=kn.to(device), v_new=vn.to(device), k_cache=kc.to(device),
                v_cache=vc.to(device), page_table=pt.to(device), page_table_host=pt, qo=qo, pl=pl,
                max_kv=max_kv, h_q=h_q, h_kv=h_kv)


def extract_pages(k_cache, v_cache, page_table_host, seqs, kv_lens):
    """CPU copy of just the pages the listed sequences use, with a compact page table."""
    pg = k_cache.shape[1]
    need = [-(-L // pg) for L in kv_lens]
    ids = torch.cat([page_table_host[s, :n].long() for s, n in zip(seqs, need)])
    kc = k_cache[ids.to(k_cache.device)].cpu()
    vc = v_cache[ids.to(v_cache.device)].cpu()
    pt = torch.full((len(seqs), max(need)), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(need):
        pt[r, :n] = torch.arange(off, off + n, dtype=torch.int32)
        off += n
    return kc, vc, pt
