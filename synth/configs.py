"""The five synthetic model configurations and their workloads.

Shapes follow the Llama architecture as the pages describe it (the pure C +
CUDA inference engine page, section 1 overview table: Llama 3.1 8B Q8_0
resident, Llama 3.1 70B with tiered caching; the SwarmKV page for the
shared-prefix fork).  Where the workload statements are silent we take these
readings: RMSNorm eps 1e-5 and fp32 unit norm gains everywhere; untied output
matrix except for the 1B shape; plain RoPE theta with no frequency scaling.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    wtype: int            # 8 = Q8_0, 4 = Q4_0
    sigma: float          # weights drawn N(0, sigma) before quantisation
    tied: bool = False
    rms_eps: float = 1e-5
    workload: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def layer_params(self) -> int:
        H, F = self.hidden, self.ffn
        return H * self.q_dim + 2 * H * self.kv_dim + self.q_dim * H + 3 * H * F

    def block_bytes(self) -> int:
        return 34 if self.wtype == 8 else 18

    def matrix_bytes(self, rows: int, cols: int) -> int:
        return rows * ((cols + 31) // 32) * self.block_bytes()


CONFIGS = {
    # 2 layers, hidden 256, 4 q heads / 2 kv heads, head_dim 64, FFN 688, vocab 1024
    "tiny": ModelConfig("tiny", 2, 256, 4, 2, 64, 688, 1024, 10000.0, 8, 0.02,
                        workload={"prompt": 16, "decode": 32}),
    # Llama-3.2-1B shape, tied embeddings
    "1b": ModelConfig("1b", 16, 2048, 32, 8, 64, 8192, 128256, 500000.0, 8, 0.02, tied=True,
                      workload={"prompt": 512, "decode": 128}),
    # Llama-3.1-8B shape, Q8_0 (headline decode workload)
    "8b": ModelConfig("8b", 32, 4096, 32, 8, 128, 14336, 128256, 500000.0, 8, 0.02,
                      workload={"ctx": [2048, 8192], "decode": 256}),
    # 8B shape, Q4_0, shared-prefix fork into 8 branches
    "fork8b": ModelConfig("fork8b", 32, 4096, 32, 8, 128, 14336, 128256, 500000.0, 4, 0.02,
                          workload={"prefix": 4096, "branches": 8, "decode": 128}),
    # Llama-3.1-70B shape, Q4_0, resident and with a 24 GB device budget
    "70b": ModelConfig("70b", 80, 8192, 64, 8, 128, 28672, 128256, 500000.0, 4, 0.01,
                       workload={"ctx": 4096, "decode": 64, "budget_bytes": 24 * 10**9}),
}


def get_config(name: str) -> ModelConfig:
    try:
        return CONFIGS[name]
    except KeyError:
        raise KeyError(f"unknown config {name!r}; known: {sorted(CONFIGS)}") from None
