"""Helpers shared by the GPU tests: device copies of a workload, one call
through the C ABI, and the parity tolerance."""
import numpy as np
import torch

from paged_kv_attention_02_gb300 import binding as b
from paged_kv_attention_02_gb300 import workloads as wl

# Tolerances: bf16 pools -- max |gpu - ref| <= 1e-2 and, per element,
# |gpu - ref| / max(|ref|, 1e-2) <= 2e-2; fp8 pools -- max |gpu - ref| <= 4e-2.
# The output is bf16, so no kernel can return ref itself: the absolute bounds
# count the error beyond the rounding of ref to the nearest bf16 (at most half
# a bf16 ulp, 2^-9 |ref|), which past |ref| = 4 alone can exceed 1e-2.
BF16_ABS, BF16_REL, REL_FLOOR, FP8_ABS = 1e-2, 2e-2, 1e-2, 4e-2


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class DevWorkload:
    def __init__(self, w: wl.Workload, device="cuda"):
        self.w = w
        self.fp8 = w.cfg.kv_dtype == wl.KV_FP8_E4M3
        self.q = bf16_tensor(w.q, device)
        if self.fp8:
            self.k = torch.from_numpy(w.k_pool).to(device)
            self.v = torch.from_numpy(w.v_pool).to(device)
            self.ks = torch.from_numpy(w.k_scales).to(device)
            self.vs = torch.from_numpy(w.v_scales).to(device)
        else:
            self.k = bf16_tensor(w.k_pool, device)
            self.v = bf16_tensor(w.v_pool, device)
            self.ks = self.vs = None
        self.table = torch.from_numpy(w.page_table).to(device)
        self.lens = torch.from_numpy(w.seq_lens).to(device)

    def run(self, q=None, table=None, lens=None, stream=None, out=None, workspace=None, window=None,
            scale=None, k=None, v=None):
        """One call through rad_attn_paged, or rad_attn_paged_window when
        `window` is given; returns (out, err_word)."""
        c = self.w.cfg
        err = torch.zeros(1, dtype=torch.int32, device=self.q.device)
        args = (self.q if q is None else q, self.k if k is None else k, self.v if v is None else v,
                self.table if table is None else table, self.lens if lens is None else lens)
        kw = dict(rows=c.rows, n_head=c.n_head, n_head_kv=c.n_head_kv,
                  head_dim=c.meta.get("head_dim", c.head_dim), page_size=c.page_size,
                  scale=c.scale if scale is None else scale, kv_dtype=c.kv_dtype, k_scales=self.ks,
                  v_scales=self.vs, out=out, workspace=workspace, err_word=err, stream=stream)
        if window is None:
            out = b.attn_paged(*args, **kw)
        else:
            out = b.attn_paged_window(*args, window=window, **kw)
        torch.cuda.synchronize()
        return out, int(err.item())


def oracle_rows(w: wl.Workload, sel=None, window=0, scale=None, page_table=None):
    import oracle
    args = w.call_args()
    if scale is not None:
        args["scale"] = scale
    return oracle.attn_paged_rows(w.q, w.k_pool, w.v_pool,
                                  w.page_table if page_table is None else page_table, w.seq_lens,
                                  sel=sel, k_scales=w.k_scales, v_scales=w.v_scales, window=window,
                                  **args)


def bf16_rounding(ref: np.ndarray) -> np.ndarray:
    """|bf16_rne(ref) - ref|: the part of any bf16 output's error that comes
    from the output format alone."""
    r = torch.from_numpy(np.ascontiguousarray(ref, dtype=np.float64))
    return (r.to(torch.bfloat16).to(torch.float64) - r).abs().numpy()


def assert_parity(gpu: np.ndarray, ref: np.ndarray, fp8: bool, what=""):
    assert gpu.shape == ref.shape, what
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    d = np.abs(gpu - ref)
    excess = d - bf16_rounding(ref)   # error beyond the output's own rounding
    if fp8:
        assert excess.max() <= FP8_ABS, f"{what}: max abs {d.max():.3e} (beyond bf16 rounding {excess.max():.3e}) > {FP8_ABS}"
    else:
        rel = d / np.maximum(np.abs(ref), REL_FLOOR)
        assert excess.max() <= BF16_ABS, f"{what}: max abs {d.max():.3e} (beyond bf16 rounding {excess.max():.3e}) > {BF16_ABS}"
        assert rel.max() <= BF16_REL, f"{what}: max rel {rel.max():.3e} > {BF16_REL}"


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy()
