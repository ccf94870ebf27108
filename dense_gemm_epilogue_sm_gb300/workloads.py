"""Seeded synthetic GEMM workloads: problem specs and input tensors.

Input generation only; no GEMM arithmetic lives here.  Both the CUDA path
(tests, benchmark) and the oracle read the tensors built here, so parity does
not depend on how they are drawn.

Recipe: a ``torch.Generator('cpu')`` seeded per workload draws, in this
order, A, B, C, bias as fp32 in storage order; 16-bit operands are the fp32
draws rounded to nearest-even.  8-bit (e4m3) operands are quantised with a
per-tensor scale s = 448 / max|x| (q = e4m3(clamp(x*s, +-448)), rounded to
nearest-even by torch) and the dequantisation factors 1/s are handed to the
GEMM as scale_a / scale_b.  Block-scaled operands (mx_float8, nv_float4)
are quantised per block of K from N(0,1) draws spread by a random power of
two per block; the factors are laid out in the 512-byte basic-block layout.

The named workloads are the five configurations the method is measured on:
a tiny exact fp16 GEMM, plain bf16 4096^3, the fused-epilogue bf16 8192^3
ReLU(0.5*A*B + C + bias), e4m3 8192^3, and odd/skinny/batched bf16 shapes.
"""
from dataclasses import dataclass, field, replace

import torch

# e2m1 (nv_float4) operands are stored as bytes, two elements per byte
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn,
      "e2m1": torch.uint8}
ESIZE = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1, "e2m1": 0.5}
SF_VEC = {"mx": 32, "nv": 16}


@dataclass
class Spec:
    name: str
    M: int
    N: int
    K: int
    batch: int = 1
    op_a: str = "N"
    op_b: str = "N"
    order_a: str = "row"
    order_b: str = "col"
    order_c: str = "row"
    order_d: str = "row"
    dtype_in: str = "bf16"
    dtype_d: str = "bf16"
    alpha: float = 1.0
    beta: float = 0.0
    act: str = "none"          # none | relu | gelu
    bias: str = "none"          # none | col | row
    dist: str = "normal"        # normal | int4 | uniform1
    bias_sigma: float = 0.1
    seed: int = 0
    pad: int = 0                # extra elements added to every leading dimension
    lda: int = 0                # 0: tight (+pad)
    ldb: int = 0
    ldc: int = 0
    ldd: int = 0
    reduce: str = "none"        # none, or a '+'-joined subset of row, col, amax
    block_scale: str = "none"   # none | mx (e4m3 data, ue8m0 scale per 32 elements of K)
                                # | nv (e2m1 data, ue4m3 scale per 16 elements of K)
    scale_d: float = 1.0        # e2m1 D (NVFP4 output): the output's global scale
    groups: int = 0             # > 0: grouped GEMM; M = rows of all groups, B and bias per group
    group_sizes: tuple = ()     # grouped: explicit rows per group (else drawn by the generator)
    notes: str = ""

    # ----------------------------------------------------------- geometry --
    def stored(self, which):
        """(rows, cols) of the stored matrix."""
        if which == "a":
            return (self.M, self.K) if self.op_a == "N" else (self.K, self.M)
        if which == "b":
            return (self.K, self.N) if self.op_b == "N" else (self.N, self.K)
        return (self.M, self.N)

    def order(self, which):
        return {"a": self.order_a, "b": self.order_b, "c": self.order_c, "d": self.order_d}[which]

    def ld(self, which):
        given = {"a": self.lda, "b": self.ldb, "c": self.ldc, "d": self.ldd}[which]
        if given:
            return given
        r, c = self.stored(which)
        tight = c if self.order(which) == "row" else r
        esz = ESIZE[self.dtype_in if which in "ab" else self.dtype_d]
        align = int(16 / esz)
        return max(align, -(-(tight + self.pad) // align) * align)

    def outer(self, which):
        r, c = self.stored(which)
        return r if self.order(which) == "row" else c

    def matrix_elems(self, which):
        return self.outer(which) * self.ld(which)

    def flops(self):
        return 2.0 * self.M * self.N * self.K * self.batch

    def algorithmic_bytes(self):
        """Each operand read once, D written once (bias and C included)."""
        e_in, e_d = ESIZE[self.dtype_in], ESIZE[self.dtype_d]
        b = self.batch * (self.M * self.K * e_in + self.K * self.N * e_in + self.M * self.N * e_d)
        if self.groups:                     # one B per group
            b += (self.groups - 1) * self.K * self.N * e_in
        if self.beta != 0:
            b += self.batch * self.M * self.N * e_d
        if self.bias != "none":
            b += 4 * (self.N if self.bias == "col" else self.M) * max(1, self.groups)
        if self.block_scale != "none":      # one byte per SV elements of K, per row of A and of B
            sv = SF_VEC[self.block_scale]
            b += self.batch * (self.M + self.N * max(1, self.groups)) * ((self.K + sv - 1) // sv)
        if self.dtype_d in ("e4m3", "e2m1"):  # output factors: one byte per 32 (MX) or 16 (NV) of a row
            sv = 32 if self.dtype_d == "e4m3" else 16
            b += self.batch * self.M * ((self.N + sv - 1) // sv)
        return int(b)


WORKLOADS = {
    "tiny_exact_fp16_256": Spec(
        "tiny_exact_fp16_256", 256, 256, 256, op_a="N", op_b="N", order_a="col", order_b="col",
        order_c="col", order_d="col", dtype_in="f16", dtype_d="f32", dist="int4", seed=0,
        notes="integer entries in [-4,4]; every sum exact in fp32"),
    "bf16_4096": Spec("bf16_4096", 4096, 4096, 4096, order_a="row", order_b="col", seed=1),
    "fused_bf16_8192": Spec(
        "fused_bf16_8192", 8192, 8192, 8192, order_a="row", order_b="col", alpha=0.5, beta=1.0,
        act="relu", bias="col", seed=2, notes="D = ReLU(0.5*A*B + 1.0*C + bias[n])"),
    "plain_bf16_8192": Spec(
        "plain_bf16_8192", 8192, 8192, 8192, order_a="row", order_b="col", seed=2,
        notes="the fused workload's GEMM alone: beta = 0, no bias, no activation"),
    "fp8_e4m3_8192": Spec(
        "fp8_e4m3_8192", 8192, 8192, 8192, order_a="row", order_b="col", dtype_in="e4m3",
        dist="uniform1", seed=3, notes="per-tensor scales folded into alpha"),
    "mxfp8_8192": Spec(
        "mxfp8_8192", 8192, 8192, 8192, order_a="row", order_b="col", dtype_in="e4m3", block_scale="mx", seed=7,
        notes="mx_float8: e4m3 data, one ue8m0 scale factor per 32 elements of K"),
    "mxfp8_to_mxfp8_8192": Spec(
        "mxfp8_to_mxfp8_8192", 8192, 8192, 8192, order_a="row", order_b="col", dtype_in="e4m3", block_scale="mx",
        dtype_d="e4m3", act="relu", seed=8,
        notes="MX in, MX out: e4m3 D with a ue8m0 factor per 32 elements of a row"),
    "nvfp4_8192": Spec(
        "nvfp4_8192", 8192, 8192, 8192, order_a="row", order_b="col", dtype_in="e2m1", block_scale="nv", seed=9,
        notes="nv_float4: e2m1 data, one ue4m3 scale factor per 16 elements of K, fp32 global scales"),
    "nvfp4_to_nvfp4_8192": Spec(
        "nvfp4_to_nvfp4_8192", 8192, 8192, 8192, order_a="row", order_b="col", dtype_in="e2m1", block_scale="nv",
        dtype_d="e2m1", act="relu", scale_d=8.0, seed=11,
        notes="NVFP4 in, NVFP4 out: e2m1 D with a ue4m3 factor per 16 elements of a row, global scale 8"),
    "grouped_16x_bf16": Spec(
        "grouped_16x_bf16", 32768, 4096, 4096, order_a="row", order_b="col", groups=16, act="relu", bias="col",
        seed=10, notes="16 groups of ragged row counts (32768 rows in all), one 4096x4096 B and bias per group"),
    "odd_1000_at": Spec(
        "odd_1000_at", 1000, 1000, 1000, op_a="T", order_a="col", order_b="col", seed=4,
        notes="A transposed: stored K x M column-major, lda = K"),
    "skinny_65536x256x4096": Spec(
        "skinny_65536x256x4096", 65536, 256, 4096, order_a="row", order_b="col", beta=1.0, seed=5,
        notes="memory-bound: A dominates the bytes"),
    "batched_32x512": Spec("batched_32x512", 512, 512, 512, batch=32, order_a="row", order_b="col", seed=6),
}


def get(name, **overrides):
    return replace(WORKLOADS[name], **overrides)


def _draw(gen, n, dist):
    if dist == "normal":
        return torch.randn(n, generator=gen, dtype=torch.float32)
    if dist == "int4":
        return torch.randint(-4, 5, (n,), generator=gen).to(torch.float32)
    if dist == "uniform1":
        return torch.rand(n, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError(dist)


def _quantise_e4m3(x):
    """Per-tensor e4m3 quantisation: returns (codes, dequantisation factor)."""
    amax = float(x.abs().max())
    s = 448.0 / amax if amax > 0 else 1.0
    s = float(torch.tensor(s, dtype=torch.float32))
    q = (x * s).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q, float(torch.tensor(1.0 / s, dtype=torch.float32))


@dataclass
class Inputs:
    spec: Spec
    A: torch.Tensor                  # flat storage, operand dtype
    B: torch.Tensor
    C: torch.Tensor = None           # flat storage, D's dtype (None when beta == 0)
    bias: torch.Tensor = None        # fp32, (batch * len) when present
    scale_a: float = 1.0
    scale_b: float = 1.0
    extras: dict = field(default_factory=dict)

    def stride(self, which):
        return self.spec.matrix_elems(which) if self.spec.batch > 1 else 0

    def bias_len(self):
        s = self.spec
        return 0 if s.bias == "none" else (s.N if s.bias == "col" else s.M)


def _sf_offsets(L, rows, sfk):
    """Byte offsets (L, rows, sfk) of the scale factors in the 512-byte
    basic-block layout: 128 rows x 4 factors per block, row r's four factors
    at (r % 32) * 16 + ((r % 128) // 32) * 4, blocks K-major, one tensor per
    batch.  Returns (offsets, tensor bytes per batch)."""
    kb, mb = (sfk + 3) // 4, (rows + 127) // 128
    r = torch.arange(rows).view(1, rows, 1)
    f = torch.arange(sfk).view(1, 1, sfk)
    l = torch.arange(L).view(L, 1, 1)
    off = ((r // 128) * kb + f // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + f % 4
    return off + l * (mb * kb * 512), mb * kb * 512


def _mx_quantise(x):
    """(L, R, K) fp32 -> (e4m3 values, ue8m0 codes (L, R, ceil(K/32))): per
    32-element block of K the shared exponent floor(log2 amax) - 8 (8 =
    exponent of e4m3's largest power of two), elements divided by it and
    rounded to e4m3, clamped to +-448."""
    L, R, K = x.shape
    sfk = (K + 31) // 32
    xp = torch.zeros(L, R, sfk * 32)
    xp[:, :, :K] = x
    blk = xp.view(L, R, sfk, 32)
    amax = blk.abs().amax(dim=3)
    e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 8,
                    torch.full_like(amax, -127.0))
    code = (e + 127).clamp(0, 254)
    scaled = (blk / torch.exp2(code - 127).unsqueeze(3)).clamp(-448.0, 448.0)
    q = scaled.to(torch.float8_e4m3fn).view(L, R, sfk * 32)[:, :, :K]
    return q, code.to(torch.uint8)


# e2m1 magnitudes by code 0..7 (sign in bit 3)
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _encode_e2m1(v):
    """fp32 -> e2m1 codes (uint8, 0..15): nearest of the grid, ties to the
    even code, magnitudes beyond 6 saturated to 6."""
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.int64)
    for i in range(7):
        t = 0.5 * (E2M1_GRID[i] + E2M1_GRID[i + 1])
        code += ((a > t) | ((a == t) & (i % 2 == 1))).to(torch.int64)
    return (code | torch.where(v < 0, 8, 0)).to(torch.uint8)


def _nv_quantise(x):
    """(L, R, K) fp32 -> (e2m1 codes, ue4m3 codes (L, R, ceil(K/16)), global
    scale g): g = amax / (448 * 6) over the tensor, a block's factor
    e4m3(amax_block / (6 g)), elements e2m1(x / (factor * g))."""
    L, R, K = x.shape
    sfk = (K + 15) // 16
    amax = float(x.abs().max())
    g = float(torch.tensor(amax / (448.0 * 6.0) if amax > 0 else 1.0, dtype=torch.float32))
    xp = torch.zeros(L, R, sfk * 16)
    xp[:, :, :K] = x
    blk = xp.view(L, R, sfk, 16)
    sf = (blk.abs().amax(dim=3) / (6.0 * g)).clamp(0.0, 448.0).to(torch.float8_e4m3fn)
    sf_val = sf.to(torch.float32) * g
    q = _encode_e2m1(torch.where(sf_val.unsqueeze(3) > 0, blk / sf_val.unsqueeze(3), torch.zeros_like(blk)))
    return q.view(L, R, sfk * 16)[:, :, :K], sf.view(torch.uint8), g


def _pack_e2m1(codes):
    """Flat e2m1 codes (one per element, storage order) -> bytes, the element
    of lower index in the low nibble."""
    c = codes.view(-1, 2)
    return (c[:, 0] | (c[:, 1] << 4)).contiguous()


def _to_storage(spec, which, logical):
    """Logical (L, R, K) operand (A: R = M; B: R = N, i.e. op(B) transposed)
    into the spec's flat storage, padding elements zero."""
    L = spec.batch
    op = spec.op_a if which == "a" else spec.op_b
    order = spec.order(which)
    ld = spec.ld(which)
    per = spec.matrix_elems(which)
    out = torch.zeros(L * per, dtype=logical.dtype)
    R, K = logical.shape[1], logical.shape[2]
    r = torch.arange(R).view(R, 1)
    k = torch.arange(K).view(1, K)
    # stored matrix: A op N is (M, K), op T is (K, M); B op N is (K, N), op T is (N, K)
    rows_first = (op == "N") if which == "a" else (op == "T")
    sr, sc = (r, k) if rows_first else (k, r)
    idx = sr * ld + sc if order == "row" else sr + sc * ld
    for l in range(L):
        out[l * per + idx.reshape(-1)] = logical[l].reshape(-1)
    return out


def _bs_operand(spec, gen, L, R):
    """One block-scaled operand of L x R rows of K: (element values (e4m3) or
    codes (e2m1) (L, R, K), factor codes (L, R, SFK), global scale)."""
    K = spec.K
    if spec.block_scale == "mx":
        sfk = (K + 31) // 32
        if spec.dist == "int4":
            # integers in [-4, 4] with factors 2^-1 .. 2^1: every sum exact in fp32
            q = torch.randint(-4, 5, (L, R, K), generator=gen).to(torch.float32).to(torch.float8_e4m3fn)
            code = torch.randint(126, 129, (L, R, sfk), generator=gen).to(torch.uint8)
        else:
            x = torch.randn(L, R, K, generator=gen, dtype=torch.float32)
            # a power of two per 32-element block spreads the scale factors
            shift = torch.randint(-4, 5, (L, R, sfk), generator=gen).to(torch.float32)
            x = x * torch.exp2(shift.repeat_interleave(32, dim=2)[:, :, :K])
            q, code = _mx_quantise(x)
        return q, code, 1.0
    sfk = (K + 15) // 16
    if spec.dist == "int4":
        # any e2m1 code with factors 0.5, 1, 2: every sum exact in fp32
        q = torch.randint(0, 16, (L, R, K), generator=gen).to(torch.uint8)
        code = torch.tensor([0x30, 0x38, 0x40], dtype=torch.uint8)[torch.randint(0, 3, (L, R, sfk), generator=gen)]
        return q, code, 1.0
    x = torch.randn(L, R, K, generator=gen, dtype=torch.float32)
    shift = torch.randint(-4, 5, (L, R, sfk), generator=gen).to(torch.float32)
    x = x * torch.exp2(shift.repeat_interleave(16, dim=2)[:, :, :K])
    return _nv_quantise(x)


# factor code of 1.0, written to the padding of a factor tensor
SF_ONE = {"mx": 127, "nv": 0x38}


def _bs_storage(spec, which, q):
    """Element values / codes (L, R, K) into the operand's storage."""
    st = _to_storage(spec, which, q)
    return _pack_e2m1(st) if spec.block_scale == "nv" else st


def _make_mx_inputs(spec, gen):
    L = spec.batch
    ops = {}
    for which, R in (("a", spec.M), ("b", spec.N)):
        q, code, _ = _bs_operand(spec, gen, L, R)
        off, per = _sf_offsets(L, R, code.shape[2])
        sf = torch.full((L * per,), SF_ONE["mx"], dtype=torch.uint8)       # padding factors: 1.0
        sf[off.reshape(-1)] = code.reshape(-1)
        ops[which] = (_bs_storage(spec, which, q), sf)
    return ops


def _make_nv_inputs(spec, gen):
    L = spec.batch
    ops = {}
    for which, R in (("a", spec.M), ("b", spec.N)):
        q, code, g = _bs_operand(spec, gen, L, R)
        off, per = _sf_offsets(L, R, code.shape[2])
        sf = torch.full((L * per,), SF_ONE["nv"], dtype=torch.uint8)       # padding factors: 1.0
        sf[off.reshape(-1)] = code.reshape(-1)
        ops[which] = (_bs_storage(spec, which, q), sf, g)
    return ops


def grouped_sfa_rows(spec, rows):
    """Row of the factor tensor of A holding each row of A, for a grouped
    block-scaled workload: every group's rows start a new 128-row block."""
    out = torch.empty(spec.M, dtype=torch.int64)
    base = 0
    for g in range(spec.groups):
        r0, r1 = int(rows[g]), int(rows[g + 1])
        out[r0:r1] = base + torch.arange(r1 - r0)
        base += 128 * ((r1 - r0 + 127) // 128)
    return out


def _make_grouped_bs_inputs(spec, gen, rows):
    """A (one matrix, factors in per-group 128-row blocks) and B (one matrix
    and factor tensor per group) of a grouped block-scaled workload."""
    one = replace(spec, groups=0, group_sizes=(), batch=1)
    per_group = replace(spec, groups=0, group_sizes=(), batch=spec.groups)
    qa, ca, ga = _bs_operand(one, gen, 1, spec.M)
    sfk = ca.shape[2]
    r_pad = 128 * ((spec.M + 127) // 128 + spec.groups)
    off, per = _sf_offsets(1, r_pad, sfk)
    sfa = torch.full((per,), SF_ONE[spec.block_scale], dtype=torch.uint8)
    covered = int(rows[-1])
    pr = grouped_sfa_rows(spec, rows)[:covered]
    sfa[off[0][pr].reshape(-1)] = ca[0][:covered].reshape(-1)
    qb, cb, gb = _bs_operand(per_group, gen, spec.groups, spec.N)
    offb, perb = _sf_offsets(spec.groups, spec.N, sfk)
    sfb = torch.full((spec.groups * perb,), SF_ONE[spec.block_scale], dtype=torch.uint8)
    sfb[offb.reshape(-1)] = cb.reshape(-1)
    return _bs_storage(one, "a", qa), _bs_storage(per_group, "b", qb), sfa, sfb, ga, gb


def group_rows_of(spec, gen):
    """Row offsets (groups + 1, int64) of a grouped workload: the given sizes,
    else weights drawn uniform in [0.25, 1.75] scaled to M rows (floors, the
    remainder to the last group)."""
    if spec.group_sizes:
        sizes = list(spec.group_sizes)
    else:
        w = torch.rand(spec.groups, generator=gen, dtype=torch.float64) * 1.5 + 0.25
        sizes = [int(x) for x in torch.floor(w / w.sum() * spec.M).tolist()]
        sizes[-1] += spec.M - sum(sizes)
    rows = [0]
    for n in sizes:
        rows.append(rows[-1] + n)
    return torch.tensor(rows, dtype=torch.int64)


def _make_grouped_inputs(spec, gen):
    rows = group_rows_of(spec, gen)
    extras = {"group_rows": rows}
    sa = sb = 1.0
    if spec.block_scale != "none":
        a, b, extras["sfa"], extras["sfb"], sa, sb = _make_grouped_bs_inputs(spec, gen, rows)
    else:
        a = _draw(gen, spec.matrix_elems("a"), spec.dist).to(DT[spec.dtype_in])
        b = _draw(gen, spec.groups * spec.matrix_elems("b"), spec.dist).to(DT[spec.dtype_in])
    C = None
    if spec.beta != 0:
        C = _draw(gen, spec.matrix_elems("c"), "normal" if spec.dist != "int4" else "int4").to(DT[spec.dtype_d])
    bias = None
    if spec.bias != "none":
        bias = torch.randn(spec.groups * spec.N, generator=gen, dtype=torch.float32) * spec.bias_sigma
    return Inputs(spec, a, b, C, bias, sa, sb, extras=extras)


def make_inputs(spec: Spec) -> Inputs:
    """Builds the storage buffers of one workload (CPU tensors).  Padding
    elements beyond each leading extent are drawn too (they are never read)."""
    gen = torch.Generator(device="cpu").manual_seed(spec.seed)
    if spec.groups:
        return _make_grouped_inputs(spec, gen)
    if spec.block_scale in ("mx", "nv"):
        if spec.block_scale == "nv":
            ops = _make_nv_inputs(spec, gen)
            sa, sb = ops["a"][2], ops["b"][2]
        else:
            ops = _make_mx_inputs(spec, gen)
            sa = sb = 1.0
        C = None
        if spec.beta != 0:
            C = _draw(gen, spec.batch * spec.matrix_elems("c"), "normal").to(DT[spec.dtype_d])
        bias = None
        if spec.bias != "none":
            n = spec.N if spec.bias == "col" else spec.M
            bias = torch.randn(spec.batch * n, generator=gen, dtype=torch.float32) * spec.bias_sigma
        return Inputs(spec, ops["a"][0], ops["b"][0], C, bias, sa, sb,
                      extras={"sfa": ops["a"][1], "sfb": ops["b"][1]})
    L = spec.batch
    out = {}
    scales = {}
    for which in ("a", "b"):
        n = L * spec.matrix_elems(which)
        x = _draw(gen, n, spec.dist)
        if spec.dtype_in == "e4m3":
            q, d = _quantise_e4m3(x)
            out[which] = q
            scales[which] = d
        else:
            out[which] = x.to(DT[spec.dtype_in])
            scales[which] = 1.0
    C = None
    if spec.beta != 0:
        C = _draw(gen, L * spec.matrix_elems("c"), "normal" if spec.dist != "int4" else "int4").to(DT[spec.dtype_d])
    bias = None
    if spec.bias != "none":
        n = spec.N if spec.bias == "col" else spec.M
        bias = (torch.randn(L * n, generator=gen, dtype=torch.float32) * spec.bias_sigma)
    return Inputs(spec, out["a"], out["b"], C, bias, scales["a"], scales["b"])


def empty_output(spec: Spec, device="cpu", fill=float("nan")):
    n = spec.batch * spec.matrix_elems("d")
    return torch.full((n,), fill, dtype=DT[spec.dtype_d], device=device)
