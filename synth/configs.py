"""Workload presets: model shapes, capacities and seeds of the synthetic runs.

Each preset names a decoder shape and the workload run on it.  Shapes follow
"bend-ml-llama 0.2.1.0, main.bend", section "The configuration" (smollm2_135m,
smollm2_1_7b) and "Llama 3.1 8B Instruct" (model card README and nest.toml:
hidden 4096, 32 query / 8 key-value heads of 128, inner 14336, 32 layers,
vocabulary 128256, untied head, theta 500000 with llama3 rope scaling).

Seeds, per preset index c: weights 1000+c, tokens 2000+c, cache values 3000+c,
uniform draws 4000+c.
"""
from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Shape:
    kv: int          # key/value heads
    g: int           # query heads per key/value head
    half: int        # half a head
    ffn: int         # MLP inner width
    layers: int
    vocab: int
    eps: float
    theta: float
    tied: bool
    llama3: bool = False
    factor: float = 8.0
    low_freq: float = 1.0
    high_freq: float = 4.0
    orig_max: float = 8192.0
    bf16: bool = True

    @property
    def hd(self):
        return 2 * self.half

    @property
    def heads(self):
        return self.kv * self.g

    @property
    def d(self):
        return self.heads * self.hd

    @property
    def kvw(self):
        return self.kv * self.hd


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    shape: Shape
    batch: int
    prompt: int          # prompt tokens prefilled (0: cache filled with synthetic values)
    steps: int           # decode steps
    cap: int             # cache capacity (positions)
    fill: int = 0        # positions of synthetic cache values (long-context preset)
    temp: float = 0.0    # 0: greedy
    top_k: int = 0       # 0: the whole vocabulary
    top_p: float = 1.0
    wstd: float = 0.02

    @property
    def seed_weights(self):
        return 1000 + self.index

    @property
    def seed_tokens(self):
        return 2000 + self.index

    @property
    def seed_kv(self):
        return 3000 + self.index

    @property
    def seed_uniform(self):
        return 4000 + self.index


TINY = Shape(kv=2, g=2, half=8, ffn=176, layers=2, vocab=256, eps=1e-5, theta=10000.0,
             tied=True, bf16=False)
SMOL135M = Shape(kv=3, g=3, half=32, ffn=1536, layers=30, vocab=49152, eps=1e-5,
                 theta=100000.0, tied=True)
SMOL1_7B = Shape(kv=32, g=1, half=32, ffn=8192, layers=24, vocab=49152, eps=1e-5,
                 theta=130000.0, tied=True)
LLAMA8B = Shape(kv=8, g=4, half=64, ffn=14336, layers=32, vocab=128256, eps=1e-5,
                theta=500000.0, tied=False, llama3=True)

WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 0, TINY, batch=1, prompt=8, steps=8, cap=16),
    "smollm2_135m": Workload("smollm2_135m", 1, SMOL135M, batch=1, prompt=128, steps=128,
                             cap=256),
    "smollm2_1_7b_b16": Workload("smollm2_1_7b_b16", 2, SMOL1_7B, batch=16, prompt=1024,
                                 steps=256, cap=1280, temp=0.8, top_k=50, top_p=0.9),
    "llama8b_b1": Workload("llama8b_b1", 3, LLAMA8B, batch=1, prompt=2048, steps=128,
                           cap=2176),
    "llama8b_b32": Workload("llama8b_b32", 3, LLAMA8B, batch=32, prompt=2048, steps=128,
                            cap=2176),
    "llama8b_long_b1": Workload("llama8b_long_b1", 4, LLAMA8B, batch=1, prompt=0, steps=64,
                                cap=131072 + 64, fill=131072, temp=0.7, top_p=0.95),
    "llama8b_long_b8": Workload("llama8b_long_b8", 4, LLAMA8B, batch=8, prompt=0, steps=64,
                                cap=32768 + 64, fill=32768, temp=0.7, top_p=0.95),
}


def weight_count(s: Shape) -> int:
    """Number of values in the weight blob (embedding, layers, final norm, untied head)."""
    layer = 2 * s.d + 2 * s.d * s.d + 2 * s.kvw * s.d + 3 * s.ffn * s.d
    return s.vocab * s.d + s.layers * layer + s.d + (0 if s.tied else s.vocab * s.d)


def shrink(s: Shape, **kw) -> Shape:
    """A copy of a shape with some fields changed (fewer layers, a smaller vocabulary...)."""
    return replace(s, **kw)
