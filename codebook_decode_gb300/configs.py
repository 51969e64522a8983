"""Model dimensions and the synthetic workloads, as plain data.

Dimensions follow the Qwen3-TTS 1.7B shapes the pages name: a 2048-wide
Talker with a codebook-0 head, a 2048->1024 small_to_mtp_projection
("Qwen3-TTS PR 5", section "What changed vs the 0.6B port") and a 1024-wide
Code Predictor that fills the other 15 codebooks ("De grens van snelheid en
kosten verleggen voor Qwen3-TTS", section "Hoe we Qwen3-TTS hebben
geoptimaliseerd"). Where the pages give no figure, the value here is the
reading stated in the design notes (Code-Predictor head_dim 128, eps 1e-6,
eos id 2048, no projection bias).
"""
from dataclasses import dataclass, field, asdict


@dataclass(frozen=True)
class Dims:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab0: int
    cp_hidden: int
    cp_layers: int
    cp_n_q_heads: int
    cp_n_kv_heads: int
    cp_head_dim: int
    cp_ffn: int
    cp_vocab: int
    n_codebooks: int = 16
    eos_id: int = 2048
    n_codes: int = 2048
    proj_bias: int = 0
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    cp_rope_theta: float = 1e6

    def as_dict(self):
        return asdict(self)


TINY = Dims(hidden=512, n_layers=2, n_q_heads=8, n_kv_heads=4, head_dim=64, ffn=1536, vocab0=2049,
            cp_hidden=256, cp_layers=1, cp_n_q_heads=4, cp_n_kv_heads=2, cp_head_dim=64, cp_ffn=768,
            cp_vocab=2048)

FULL = Dims(hidden=2048, n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128, ffn=6144, vocab0=3072,
            cp_hidden=1024, cp_layers=5, cp_n_q_heads=16, cp_n_kv_heads=8, cp_head_dim=128, cp_ffn=3072,
            cp_vocab=2048)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: batch, prefix lengths, frames, sampling."""
    name: str
    dims: Dims
    batch: int
    prefix: tuple          # ("fixed", n) or ("uniform", lo, hi)
    offset: tuple          # ("fixed", 0) or ("uniform", lo, hi): frames already generated
    frames: int
    temperature: float
    top_k: int
    rep_penalty: float
    shuffle_pages: bool
    int8: bool
    seed: int              # weights seed = 1000 + seed, data seed = 2000 + seed


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 1, ("fixed", 32), ("fixed", 0), 16, 0.0, 1, 1.0, False, False, 0),
    "full_b1": Workload("full_b1", FULL, 1, ("fixed", 128), ("fixed", 0), 64, 0.9, 50, 1.05, True, False, 1),
    # full widths with 2 Talker layers: a small case for profiler captures
    "full2l_b1": Workload("full2l_b1", Dims(**{**FULL.as_dict(), "n_layers": 2}), 1, ("fixed", 128), ("fixed", 0),
                          64, 0.9, 50, 1.05, True, False, 1),
    "full_b8": Workload("full_b8", FULL, 8, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True,
                        False, 2),
    "full_b32": Workload("full_b32", FULL, 32, ("uniform", 100, 1000), ("uniform", 0, 200), 256, 0.9, 50, 1.05,
                         True, False, 3),
    # full widths with 2 Talker layers at B = 32: the tensor-path small case for profiler captures
    "full2l_b32": Workload("full2l_b32", Dims(**{**FULL.as_dict(), "n_layers": 2}), 32, ("uniform", 100, 1000),
                           ("uniform", 0, 200), 256, 0.9, 50, 1.05, True, False, 3),
    "int8_b1": Workload("int8_b1", FULL, 1, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True, True, 4),
    "int8_b32": Workload("int8_b32", FULL, 32, ("uniform", 64, 512), ("fixed", 0), 128, 0.9, 50, 1.05, True,
                         True, 4),
}

PAGE_SIZE = 16
MAX_BATCH = 32
