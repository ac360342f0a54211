"""The five synthetic Engram workloads, named by what they are.

Every field is a plain number or string; nothing here computes any part of the
Engram layer.  The workloads stand in for the runs described on the pages:

* ``tiny_f32``          -- B=1, T=64, V=1000 -> 770, N=3, K=2, 16-dim fp32 rows, d=64.
* ``prefill_bf16``      -- B=1, T=4096, V=129280, N=3, K=8, 64-dim bf16 rows,
                           d=1024, two independent layers (ids 1 and 15).  This mirrors
                           the demo hyper-parameters of the Ascend RecSDK Engram blog
                           (ai6s.net), section "测试结果": seq 4096, max n-gram 3,
                           8 heads per n-gram, 512 dims per n-gram, 10342400 rows,
                           Engram layers 1 and 15.
* ``decode_bf16``       -- the prefill tables and weights; B=256 sequences, one new
                           token each after a 32-token prefix.
* ``int8_host``         -- B=64, T=2048, ~40M int8 rows + fp16 per-row scale per layer,
                           table rows in pinned host memory read over UVA.
* ``multibranch_n4``    -- B=8, T=8192, d=4096, M=4 hyper-connection branches, N=4,
                           24 bf16 tables near 1.5M rows each.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # 1-based position in the list below; feeds the seed
    B: int
    T: int
    V: int                     # raw vocabulary
    V_proj: int                # canonical vocabulary after projection
    N: int                     # max n-gram order (orders 2..N)
    K: int                     # hash heads per order
    row_dim: int               # elements per table row
    d: int                     # hidden size
    M: int                     # hyper-connection branches
    conv_w: int
    conv_dil: int
    table_dtype: str           # "f32" | "bf16" | "i8"
    act_dtype: str             # "f32" | "bf16"
    prime_target: int          # primes are the first R primes >= this
    layers: Tuple[int, ...]    # layer ids; each layer has its own tables/weights
    zipf_s: float
    span_len: int              # length of the repeated motif (0 = none)
    span_copies: int           # non-overlapping copies of it per sequence
    prefix_len: int = 0        # decode only: tokens already seen per sequence
    table_std: float = 0.02
    h_std: float = 1.0
    w_std: float = 0.0         # 0 -> 1/sqrt(d_mem)
    norm_std: float = 0.1      # RMSNorm weights are 1 + N(0, norm_std)
    conv_std: float = 0.5
    eps: float = 1e-6
    weight_seed_index: int = 0  # 0 -> use own index; else share another workload's weights
    table_in_host: bool = False

    @property
    def R(self) -> int:
        return (self.N - 1) * self.K

    @property
    def d_mem(self) -> int:
        return self.R * self.row_dim

    @property
    def ntok(self) -> int:
        return self.B * self.T

    @property
    def base_seed(self) -> int:
        return 20260112 + self.index

    @property
    def weight_seed(self) -> int:
        return 20260112 + (self.weight_seed_index or self.index)

    @property
    def multiplier_count(self) -> int:
        # one multiplier per (order n, head k, window slot i), i < n
        return sum(self.K * n for n in range(2, self.N + 1))

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (for smaller test cases)."""
        return replace(self, **kw)


TINY_F32 = Workload(
    name="tiny_f32", index=1, B=1, T=64, V=1000, V_proj=770, N=3, K=2, row_dim=16,
    d=64, M=1, conv_w=4, conv_dil=3, table_dtype="f32", act_dtype="f32",
    prime_target=1009, layers=(0,), zipf_s=1.1, span_len=8, span_copies=3,
    w_std=0.125,
)

PREFILL_BF16 = Workload(
    name="prefill_bf16", index=2, B=1, T=4096, V=129280, V_proj=99546, N=3, K=8,
    row_dim=64, d=1024, M=1, conv_w=4, conv_dil=3, table_dtype="bf16",
    act_dtype="bf16", prime_target=646400, layers=(1, 15), zipf_s=1.1,
    span_len=16, span_copies=13,
)

DECODE_BF16 = Workload(
    name="decode_bf16", index=3, B=256, T=1, V=129280, V_proj=99546, N=3, K=8,
    row_dim=64, d=1024, M=1, conv_w=4, conv_dil=3, table_dtype="bf16",
    act_dtype="bf16", prime_target=646400, layers=(1, 15), zipf_s=1.1,
    span_len=0, span_copies=0, prefix_len=32, weight_seed_index=2,
)

INT8_HOST = Workload(
    name="int8_host", index=4, B=64, T=2048, V=129280, V_proj=99546, N=3, K=8,
    row_dim=64, d=1024, M=1, conv_w=4, conv_dil=3, table_dtype="i8",
    act_dtype="bf16", prime_target=2500000, layers=(1,), zipf_s=1.1,
    span_len=16, span_copies=7, table_in_host=True,
)

MULTIBRANCH_N4 = Workload(
    name="multibranch_n4", index=5, B=8, T=8192, V=129280, V_proj=99546, N=4, K=8,
    row_dim=64, d=4096, M=4, conv_w=4, conv_dil=4, table_dtype="bf16",
    act_dtype="bf16", prime_target=1500000, layers=(1,), zipf_s=1.05,
    span_len=32, span_copies=26,
)

ALL = (TINY_F32, PREFILL_BF16, DECODE_BF16, INT8_HOST, MULTIBRANCH_N4)
BY_NAME = {w.name: w for w in ALL}
