"""Seeded synthetic inputs for MLA decode (shared by the tests, the smoke check
and the benchmark; holds no attention arithmetic).

The shapes follow the problem statement of kernelbot-amd-mixed-mla-675627
("MLA decode kernel -- submission template", the docstring's input tuple):
``q [total_q, 16, 576]`` bf16, a KV cache ``[total_kv, 1, 576]`` in bf16, fp8
e4m3 with one per-tensor scale, or mxfp4 (fp4x2 ``[total_kv, 1, 288]`` plus
e8m0 block scales), and int32 ``qo_indptr`` / ``kv_indptr``.

Quantisers (input preparation, not part of the decode path):
  * fp8: the per-tensor rule of that page's ``quantize_fp8`` --
    scale = max(amax, 1e-12) / 448, codes = clamp(x / scale, +-448) cast to
    e4m3fn (round to nearest even).
  * mxfp4: OCP MX v1.0 -- per 32-element block, X = floor(log2(amax)) - 2
    clamped to [-127, 127], e8m0 byte = X + 127, elements = x / 2^X rounded to
    the nearest e2m1 value (ties to the even code), saturating at +-6; element
    2i in the low nibble of byte i, 2i+1 in the high nibble.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import BF16, D_QK, D_V, FP8_E4M3, HEADS, MX_BLOCK, MXFP4  # noqa: F401  (sizes and format codes)

FP8_MAX = 448.0
DTYPE_NAMES = {BF16: "bf16", FP8_E4M3: "fp8_e4m3", MXFP4: "mxfp4"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    q_len: int
    kv_len: int          # per segment; ignored when ragged
    q_dtype: int
    kv_dtype: int
    ragged_max: int = 0  # > 0: kv_len_b ~ U[1, ragged_max]
    seed: int = 0

    def describe(self) -> str:
        kv = f"U[1,{self.ragged_max}]" if self.ragged_max else str(self.kv_len)
        return (f"batch {self.batch} x q_len {self.q_len}, kv_len {kv}, q {DTYPE_NAMES[self.q_dtype]}, "
                f"kv {DTYPE_NAMES[self.kv_dtype]}")


# The five benchmark workloads (sizes from the pages' shape grid; seeds fixed).
WORKLOADS = {
    "bf16_bs4_kv1024": Workload("bf16_bs4_kv1024", 4, 1, 1024, BF16, BF16),
    "fp8kv_bs32_kv8192": Workload("fp8kv_bs32_kv8192", 32, 1, 8192, BF16, FP8_E4M3),
    "a8w8_bs64_kv1024": Workload("a8w8_bs64_kv1024", 64, 1, 1024, FP8_E4M3, FP8_E4M3),
    "fp8kv_bs256_kv8192": Workload("fp8kv_bs256_kv8192", 256, 1, 8192, BF16, FP8_E4M3),
    "mxfp4_bs128_ragged16384": Workload("mxfp4_bs128_ragged16384", 128, 1, 0, BF16, MXFP4,
                                        ragged_max=16384),
}


@dataclasses.dataclass
class Inputs:
    """Device (or host) tensors in the library's layouts."""
    q: torch.Tensor            # bf16 [total_q,16,576] or uint8 e4m3 codes
    q_scale: torch.Tensor | None   # float32 [1] when q is fp8
    kv: torch.Tensor           # bf16 [total_kv,576] | uint8 [total_kv,576] | uint8 [total_kv,288]
    kv_scale: torch.Tensor | None  # float32 [1] (fp8) | uint8 [total_kv,18] (mxfp4) | None
    qo_indptr: torch.Tensor    # int32 [batch+1]
    kv_indptr: torch.Tensor    # int32 [batch+1]
    q_dtype: int
    kv_dtype: int

    @property
    def batch(self) -> int:
        return self.qo_indptr.numel() - 1

    @property
    def total_q(self) -> int:
        return self.q.shape[0]

    @property
    def total_kv(self) -> int:
        return self.kv.shape[0]

    def kv_bytes(self) -> int:
        n = self.kv.numel() * self.kv.element_size()
        if self.kv_dtype == MXFP4:
            n += self.kv_scale.numel()
        return n


def quantize_fp8_per_tensor(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-tensor e4m3fn quantisation: returns (uint8 codes, float32 [1] scale)."""
    amax = x.abs().amax().float().clamp(min=1e-12)
    scale = (amax / FP8_MAX).float()
    codes = (x.float() / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale.reshape(1)


def quantize_mxfp4(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """OCP MX fp4 (e2m1 + e8m0 per 32) of x [rows, D]: returns (uint8 [rows, D/2], uint8 [rows, D/32])."""
    rows, d = x.shape
    assert d % MX_BLOCK == 0
    xb = x.float().reshape(rows, d // MX_BLOCK, MX_BLOCK)
    amax = xb.abs().amax(dim=-1)
    # floor(log2(amax)) exactly, via frexp: amax = m * 2^e with m in [0.5, 1)
    _, e = torch.frexp(amax)
    xexp = (e.to(torch.int32) - 1) - 2
    xexp = torch.where(amax > 0, xexp, torch.full_like(xexp, -127)).clamp(-127, 127)
    scale_codes = (xexp + 127).to(torch.uint8)
    scaled = xb * torch.pow(2.0, -xexp.float()).unsqueeze(-1)
    mag = scaled.abs()
    # nearest e2m1 magnitude (0,.5,1,1.5,2,3,4,6); ties go to the even code
    code = ((mag > 0.25).to(torch.int32) + (mag >= 0.75).to(torch.int32) + (mag > 1.25).to(torch.int32)
            + (mag >= 1.75).to(torch.int32) + (mag > 2.5).to(torch.int32) + (mag >= 3.5).to(torch.int32)
            + (mag > 5.0).to(torch.int32))
    sign = ((scaled < 0) & (code > 0)).to(torch.int32) << 3
    nib = (code | sign).reshape(rows, d)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).to(torch.uint8)
    return packed, scale_codes.reshape(rows, d // MX_BLOCK)


def make_lengths(w: Workload) -> list[int]:
    if w.ragged_max:
        g = torch.Generator(device="cpu").manual_seed(w.seed)
        return (torch.randint(1, w.ragged_max + 1, (w.batch,), generator=g)).tolist()
    return [w.kv_len] * w.batch


def make_inputs(w: Workload, device: str | torch.device = "cpu", *, kv_lens: list[int] | None = None,
                q_lens: list[int] | None = None) -> Inputs:
    """Seeded inputs for workload w on `device` (values ~N(0,1) before quantisation).
    kv_lens / q_lens override the per-segment lengths (edge-case tests)."""
    device = torch.device(device)
    kv_lens = list(kv_lens) if kv_lens is not None else make_lengths(w)
    q_lens = list(q_lens) if q_lens is not None else [w.q_len] * len(kv_lens)
    assert len(q_lens) == len(kv_lens)
    qo = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    kvp = torch.tensor([0] + list(np.cumsum(kv_lens)), dtype=torch.int32)
    total_q, total_kv = int(qo[-1]), int(kvp[-1])
    g = torch.Generator(device=device).manual_seed(w.seed + 1)
    qf = torch.randn((total_q, HEADS, D_QK), generator=g, device=device, dtype=torch.float32)
    if w.q_dtype == BF16:
        q, q_scale = qf.to(torch.bfloat16), None
    else:
        q, q_scale = quantize_fp8_per_tensor(qf)
    del qf
    kvf = torch.randn((total_kv, D_QK), generator=g, device=device, dtype=torch.float32)
    if w.kv_dtype == BF16:
        kv, kv_scale = kvf.to(torch.bfloat16), None
    elif w.kv_dtype == FP8_E4M3:
        kv, kv_scale = quantize_fp8_per_tensor(kvf)
    else:
        kv, kv_scale = quantize_mxfp4(kvf)
    del kvf
    return Inputs(q=q.contiguous(), q_scale=q_scale, kv=kv.contiguous(), kv_scale=kv_scale,
                  qo_indptr=qo.to(device), kv_indptr=kvp.to(device), q_dtype=w.q_dtype,
                  kv_dtype=w.kv_dtype)


def to_host_codes(inp: Inputs, segments: list[int] | None = None) -> dict:
    """Raw codes as numpy (what the oracle reads). With `segments`, only those batch
    entries are kept and the indptrs are re-based; `token_map` gives the original
    token index of each kept token."""
    qo = inp.qo_indptr.cpu().numpy().astype(np.int64)
    kvp = inp.kv_indptr.cpu().numpy().astype(np.int64)
    segs = list(range(inp.batch)) if segments is None else list(segments)
    q_bits = inp.q.view(torch.int16) if inp.q_dtype == BF16 else inp.q
    kv_bits = inp.kv.view(torch.int16) if inp.kv_dtype == BF16 else inp.kv
    q_parts, kv_parts, sc_parts, tok = [], [], [], []
    new_qo, new_kv = [0], [0]
    for b in segs:
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(kvp[b]), int(kvp[b + 1])
        q_parts.append(q_bits[q0:q1].cpu().numpy())
        kv_parts.append(kv_bits[k0:k1].cpu().numpy())
        if inp.kv_dtype == MXFP4:
            sc_parts.append(inp.kv_scale[k0:k1].cpu().numpy())
        tok.extend(range(q0, q1))
        new_qo.append(new_qo[-1] + (q1 - q0))
        new_kv.append(new_kv[-1] + (k1 - k0))
    qdt = np.uint16 if inp.q_dtype == BF16 else np.uint8
    kdt = np.uint16 if inp.kv_dtype == BF16 else np.uint8
    q_np = np.concatenate(q_parts).view(qdt) if q_parts else np.zeros((0, HEADS, D_QK), qdt)
    kv_np = np.concatenate(kv_parts).view(kdt) if kv_parts else np.zeros((0,) + tuple(inp.kv.shape[1:]), kdt)
    if inp.kv_dtype == FP8_E4M3:
        kv_scale = float(inp.kv_scale.cpu()[0])
    elif inp.kv_dtype == MXFP4:
        kv_scale = (np.concatenate(sc_parts) if sc_parts
                    else np.zeros((0, D_QK // MX_BLOCK), np.uint8))
    else:
        kv_scale = None
    return dict(q=q_np, q_dtype=inp.q_dtype,
                q_scale=None if inp.q_scale is None else float(inp.q_scale.cpu()[0]),
                kv=kv_np, kv_dtype=inp.kv_dtype, kv_scale=kv_scale,
                qo_indptr=np.array(new_qo, np.int32), kv_indptr=np.array(new_kv, np.int32),
                token_map=np.array(tok, np.int64))


def sm_scale_default() -> float:
    return 1.0 / math.sqrt(D_QK)


@dataclasses.dataclass
class PagedInputs:
    """A paged fp8 KV cache: a pool of pages and a page table (int32, device)."""
    q: torch.Tensor
    q_scale: torch.Tensor | None
    kv_pages: torch.Tensor          # uint8 e4m3 codes [num_pages, page_size, 576]
    kv_scale: torch.Tensor          # float32 [1]
    qo_indptr: torch.Tensor
    page_indptr: torch.Tensor       # [batch + 1]
    page_indices: torch.Tensor      # [page_indptr[-1]]
    last_page_len: torch.Tensor     # [batch]
    page_size: int
    total_kv: int                   # logical rows, the sum of the segment lengths
    q_dtype: int
    kv_dtype: int = FP8_E4M3

    @property
    def batch(self) -> int:
        return self.qo_indptr.numel() - 1

    @property
    def total_q(self) -> int:
        return self.q.shape[0]

    @property
    def num_pages(self) -> int:
        return self.kv_pages.shape[0]


def make_paged_inputs(w: Workload, device: str | torch.device = "cpu", *, kv_lens: list[int] | None = None,
                      q_lens: list[int] | None = None, page_size: int = 1, spare_pages: int = 0,
                      lengths_as_last: bool = False) -> PagedInputs:
    """Seeded paged inputs: q as make_inputs, a pool of ceil(len/page_size) pages per
    segment plus `spare_pages` unused ones (values ~N(0,1), one per-tensor fp8 scale),
    handed out in a random order so a segment's pages are scattered over the pool.
    With page_size 1 and lengths_as_last, last_page_len holds the segment lengths
    (the argument form of kernelbot-amd-mixed-mla-753817's paged call); otherwise
    each segment's last page holds the remaining rows."""
    device = torch.device(device)
    kv_lens = list(kv_lens) if kv_lens is not None else make_lengths(w)
    base = make_inputs(dataclasses.replace(w, kv_dtype=BF16), device, kv_lens=[0] * len(kv_lens), q_lens=q_lens)
    npages = [(n + page_size - 1) // page_size for n in kv_lens]
    used = int(sum(npages))
    num_pages = used + spare_pages
    g = torch.Generator(device="cpu").manual_seed(w.seed + 2)
    order = torch.randperm(num_pages, generator=g).to(torch.int32)
    page_indices = order[:used].contiguous()
    page_indptr = torch.tensor([0] + list(np.cumsum(npages)), dtype=torch.int32)
    if page_size == 1 and lengths_as_last:
        last = list(kv_lens)
    else:
        last = [n - (p - 1) * page_size if p > 0 else page_size for n, p in zip(kv_lens, npages)]
    gk = torch.Generator(device=device).manual_seed(w.seed + 3)
    kvf = torch.randn((max(num_pages, 1) * page_size, D_QK), generator=gk, device=device, dtype=torch.float32)
    codes, scale = quantize_fp8_per_tensor(kvf)
    del kvf
    pool = codes[: num_pages * page_size].reshape(num_pages, page_size, D_QK).contiguous()
    return PagedInputs(q=base.q, q_scale=base.q_scale, kv_pages=pool, kv_scale=scale, qo_indptr=base.qo_indptr,
                       page_indptr=page_indptr.to(device), page_indices=page_indices.to(device),
                       last_page_len=torch.tensor(last, dtype=torch.int32).to(device), page_size=page_size,
                       total_kv=int(sum(kv_lens)), q_dtype=w.q_dtype)
