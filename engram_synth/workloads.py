"""The five synthetic Engram workloads, as sizes and input recipes.

Names follow the DeepSeek-V4.1 config fields (engram_layer_ids,
engram_max_ngram_size, engram_n_heads, engram_head_dim, engram_vocab_size,
engram_compressed_vocab_size, hidden_size, hc_mult, rms_norm_eps) that the
vLLM ``EngramLayout`` class and the NeMo ``DeepseekV41NgramHash`` class read.
Nothing here derives a layout; sizes that follow from the layout (primes,
table rows) are computed by whoever consumes a workload.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layer_ids: tuple            # engram_layer_ids (decoder layer numbers)
    max_ngram: int              # n-gram sizes 2..max_ngram
    n_heads: int                # hash heads per n-gram size
    head_dim: int               # width of one table row
    vocab_size: int             # engram_vocab_size: prime search starts above vocab_size - 1
    raw_vocab: int              # tokenizer ids
    compressed_vocab: int       # engram_compressed_vocab_size
    hidden: int                 # hidden_size (H)
    hc: int                     # hc_mult (highway streams)
    table_format: str           # "bf16" | "fp8" | "q2k"
    seq_lens: tuple             # new tokens per sequence
    id_dist: str = "uniform"    # raw id distribution: "uniform" | "zipf"
    zipf_alpha: float = 1.1
    map_kind: str = "surjection"  # token_map: "surjection" | "permutation"
    docs_per_seq: tuple | None = None   # (lo, hi) documents per sequence, None = no sequence_ids
    mask_frac: float = 0.0              # fraction of positions with token_mask false
    lookback: bool = False              # pass max_ngram-1 prior compressed ids per sequence
    lookback_dead_frac: float = 0.0     # fraction of lookback entries marked unavailable (-1)
    pad_token_id: int = 0               # raw id whose compressed id pads the window
    eps: float = 1e-6
    clamp: float = 1e-6
    table_std: float = 0.02
    wkv_std: float = 0.02
    qk_std: float = 0.1
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def layers(self) -> int:
        return len(self.layer_ids)

    @property
    def cols(self) -> int:
        return (self.max_ngram - 1) * self.n_heads

    @property
    def K(self) -> int:
        return self.cols * self.head_dim

    @property
    def N(self) -> int:
        return self.hidden * (self.hc + 1)

    def with_tokens(self, seq_lens: tuple) -> "Workload":
        return replace(self, seq_lens=tuple(seq_lens))


_DECODE = Workload(
    name="decode_fp8_t256",
    seed=1,
    layer_ids=(1,),
    max_ngram=4,
    n_heads=8,
    head_dim=256,
    vocab_size=1 << 20,
    raw_vocab=163840,
    compressed_vocab=131072,
    hidden=4096,
    hc=4,
    table_format="fp8",
    seq_lens=(1,) * 256,
    id_dist="zipf",
    lookback=True,
)

WORKLOADS = {
    # 1 sequence of 64 uniform raw ids over 4096, 1024 compressed ids,
    # n-grams 2..3 x 4 heads, primes just above 4000, bf16 rows of 64.
    "tiny_bf16": Workload(
        name="tiny_bf16",
        seed=0,
        layer_ids=(1,),
        max_ngram=3,
        n_heads=4,
        head_dim=64,
        vocab_size=4001,
        raw_vocab=4096,
        compressed_vocab=1024,
        hidden=256,
        hc=4,
        table_format="bf16",
        seq_lens=(64,),
    ),
    # 256 sequences x 1 new token, 3 lookback ids each, Zipf(1.1) raw ids,
    # 24 heads (sizes 2..4 x 8), primes above 2^20, FP8+E8M0 rows of 256.
    "decode_fp8_t256": _DECODE,
    # Same, with 10% of lookback entries unavailable (correctness only).
    "decode_fp8_t256_deadlb": replace(_DECODE, name="decode_fp8_t256_deadlb",
                                      seed=11, lookback_dead_frac=0.10),
    # 8 x 4096 Zipf ids, 3-6 documents per sequence, 5% masked positions.
    "prefill_fp8_t32768": replace(
        _DECODE,
        name="prefill_fp8_t32768",
        seed=2,
        seq_lens=(4096,) * 8,
        docs_per_seq=(3, 6),
        mask_frac=0.05,
        lookback=False,
    ),
    # Two engram layers (1 and 14), primes above 2^19, Q2_K rows, 4 x 2048 tokens.
    "q2k_t8192": replace(
        _DECODE,
        name="q2k_t8192",
        seed=3,
        layer_ids=(1, 14),
        vocab_size=1 << 19,
        table_format="q2k",
        seq_lens=(2048,) * 4,
        lookback=False,
    ),
    # Large table: primes above 2^23 (about 53 GB FP8+E8M0), hidden 7168,
    # uniform compressed ids (token_map a permutation).  T is swept.
    "large_fp8_t16384": replace(
        _DECODE,
        name="large_fp8_t16384",
        seed=4,
        vocab_size=1 << 23,
        raw_vocab=131072,
        compressed_vocab=131072,
        hidden=7168,
        seq_lens=(16384,),
        id_dist="uniform",
        map_kind="permutation",
        lookback=False,
    ),
}
# Small cases for the FP8 operand variant: the tiny config's token recipe (64 uniform ids, one
# sequence, primes just above 4000) with FP8+E8M0 rows of 256 (K = 8 * 256 = 2048), and a
# two-layer version of the decode step (layers 1 and 14) for the per-layer loop.
WORKLOADS["tiny_fp8"] = replace(WORKLOADS["tiny_bf16"], name="tiny_fp8", seed=5, head_dim=256,
                                table_format="fp8")
WORKLOADS["decode_fp8_t256_2layer"] = replace(_DECODE, name="decode_fp8_t256_2layer", seed=6,
                                              layer_ids=(1, 14))
for _t in (1, 64, 1024):
    WORKLOADS[f"large_fp8_t{_t}"] = replace(
        WORKLOADS["large_fp8_t16384"], name=f"large_fp8_t{_t}", seq_lens=(_t,))


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
