"""The five synthetic workloads: shapes, storage types and value distributions.

Each tensor is drawn from its own generator stream under seed 0: x from
stream 0, w from stream 1, dy from stream 2, b from stream 3.  ``N(m, s)`` means mean m and
standard deviation s.  Nothing here computes any part of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import NORMAL, UNIFORM

SEED = 0
STREAM_X, STREAM_W, STREAM_DY, STREAM_B = 0, 1, 2, 3


@dataclass(frozen=True)
class Dist:
    kind: int      # NORMAL or UNIFORM
    a: float       # mean (normal) or low end (uniform)
    b: float       # standard deviation (normal) or high end (uniform)


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                  # "ws" (weighted sum), "silu" (scaled SiLU), "softmax",
                             # "rmsnorm" or "layernorm"
    dtype: str               # storage type of x, dy, y, dx: "f32" | "f16" | "bf16"
    N: int                   # rows (ws) or leading extent (silu)
    D: int                   # features (ws) or trailing extent (silu)
    x: Dist
    dy: Dist
    w: Dist | None = None    # ws, norms: w[D] in binary32
    b: Dist | None = None    # layernorm: b[D] in binary32
    eps: float = 0.0         # norms: the binary32 eps under the square root
    w_scalar: float | None = None  # silu: the scalar w in binary32
    block_n: int = 0         # rows per partial tile (0: the library chooses)
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return self.N * self.D


WORKLOADS = {
    "c1": Workload("c1", "ws", "f32", 100, 64, x=Dist(NORMAL, 0.0, 1.0), w=Dist(NORMAL, 0.0, 1.0),
                   dy=Dist(NORMAL, 0.0, 1.0), block_n=32,
                   note="weighted sum, fp32 x[100,64]; 32-row tiles give a [4,64] partial buffer"),
    "c2": Workload("c2", "silu", "f16", 8192, 4096, x=Dist(NORMAL, 0.0, 2.0), w_scalar=0.75,
                   dy=Dist(NORMAL, 0.0, 1.0),
                   note="scaled SiLU, fp16 x[8192,4096] ~N(0,2), w=0.75, scalar dw over 33.5M elements"),
    "c3": Workload("c3", "ws", "bf16", 1 << 20, 1024, x=Dist(NORMAL, 0.0, 1.0),
                   w=Dist(NORMAL, 0.0, 1.0 / 32.0), dy=Dist(NORMAL, 0.0, 1.0),
                   note="weighted sum, bf16 x[1048576,1024], w ~N(0,1/sqrt(1024))"),
    "c4": Workload("c4", "ws", "f16", 1 << 24, 64, x=Dist(UNIFORM, -1.0, 1.0),
                   w=Dist(NORMAL, 0.0, 1.0), dy=Dist(NORMAL, 0.0, 1.0),
                   note="tall-skinny weighted sum, fp16 x[16777216,64] ~U(-1,1)"),
    "c5": Workload("c5", "ws", "f32", 4096, 65536, x=Dist(NORMAL, 0.0, 1.0),
                   w=Dist(NORMAL, 0.0, 1.0 / 256.0), dy=Dist(NORMAL, 0.0, 1.0),
                   note="wide weighted sum, fp32 x[4096,65536], w ~N(0,1/256)"),
    # measurement case of the softmax backward (rows of 4096, as in the
    # softmax example of the VJP essay); not part of the default benchmark step
    "s1": Workload("s1", "softmax", "bf16", 65536, 4096, x=Dist(NORMAL, 0.0, 2.0),
                   dy=Dist(NORMAL, 0.0, 1.0),
                   note="row softmax, bf16 x[65536,4096] ~N(0,2), dy ~N(0,1)"),
    # measurement cases of the norm backward: B·T = 65,536 token rows of
    # width 4096 (the RMSNorm dw example of the backward-grid essay, and
    # LayerNorm from the VJP essay); not part of the default benchmark step
    "n1": Workload("n1", "rmsnorm", "bf16", 65536, 4096, x=Dist(NORMAL, 0.0, 1.0),
                   w=Dist(NORMAL, 1.0, 0.1), dy=Dist(NORMAL, 0.0, 1.0), eps=2.0 ** -17,
                   note="RMSNorm, bf16 x[65536,4096] ~N(0,1), w ~N(1,0.1), eps 2^-17"),
    "n2": Workload("n2", "layernorm", "bf16", 65536, 4096, x=Dist(NORMAL, 0.5, 1.0),
                   w=Dist(NORMAL, 1.0, 0.1), b=Dist(NORMAL, 0.0, 0.1), dy=Dist(NORMAL, 0.0, 1.0),
                   eps=2.0 ** -17,
                   note="LayerNorm, bf16 x[65536,4096] ~N(0.5,1), w ~N(1,0.1), b ~N(0,0.1), eps 2^-17"),
    # wide rows, split over thread-block clusters: a vocabulary-sized softmax
    # (131,072 columns) and norms over a hidden size of 16,384
    "s2": Workload("s2", "softmax", "bf16", 4096, 131072, x=Dist(NORMAL, 0.0, 2.0),
                   dy=Dist(NORMAL, 0.0, 1.0),
                   note="row softmax, bf16 x[4096,131072] ~N(0,2), dy ~N(0,1)"),
    # softmax rows of an odd width (a GPT-2-sized vocabulary of 50,257: rows
    # read as the 16-byte chunks that cover them) and fp32 rows wider than the
    # cluster rows hold (two passes)
    "s3": Workload("s3", "softmax", "bf16", 8192, 50257, x=Dist(NORMAL, 0.0, 2.0),
                   dy=Dist(NORMAL, 0.0, 1.0),
                   note="row softmax, bf16 x[8192,50257] ~N(0,2), dy ~N(0,1)"),
    "s4": Workload("s4", "softmax", "f32", 2048, 262144, x=Dist(NORMAL, 0.0, 2.0),
                   dy=Dist(NORMAL, 0.0, 1.0),
                   note="row softmax, fp32 x[2048,262144] ~N(0,2), dy ~N(0,1)"),
    "n3": Workload("n3", "rmsnorm", "bf16", 16384, 16384, x=Dist(NORMAL, 0.0, 1.0),
                   w=Dist(NORMAL, 1.0, 0.1), dy=Dist(NORMAL, 0.0, 1.0), eps=2.0 ** -17,
                   note="RMSNorm, bf16 x[16384,16384] ~N(0,1), w ~N(1,0.1), eps 2^-17"),
    "n4": Workload("n4", "layernorm", "bf16", 16384, 16384, x=Dist(NORMAL, 0.5, 1.0),
                   w=Dist(NORMAL, 1.0, 0.1), b=Dist(NORMAL, 0.0, 0.1), dy=Dist(NORMAL, 0.0, 1.0),
                   eps=2.0 ** -17,
                   note="LayerNorm, bf16 x[16384,16384] ~N(0.5,1), w ~N(1,0.1), b ~N(0,0.1), eps 2^-17"),
}
