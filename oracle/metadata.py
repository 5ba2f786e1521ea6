"""Oracle for the step metadata of the paged-KV path -- TEST INFRASTRUCTURE ONLY.

Plain Python loops over small inputs; only tests and the benchmark's CPU
legs use it.  What it computes follows nano-vllm as described on the page
"13. 读一个最小推理引擎：nano-vllm":

* every step computes the tokens of a sequence from num_cached_tokens onward
  ("第二站：一个请求的状态"); a prefill feeds only those tokens and a decode
  step feeds the one new token ("第五站：执行准备与 KV 容量");
* a token at logical position p goes to slot
  block_table[p // block_size] * block_size + p % block_size ("第五站", slot
  mapping);
* the varlen attention calls take cumulative sequence lengths of the new
  tokens (queries) and of all tokens (keys) ("第六站：注意力层").

* a CUDA-graph step is padded to its captured batch size with rows whose
  slot is -1 and whose context length is 0 ("第五站", CUDA Graph paragraph);
  here such a pad row is a sequence with c_i = L_i = 0: it adds no new
  tokens and no keys, its context length is 0 and its table row is -1.

Inputs per sequence i: its block table (list of physical block ids),
num_cached c_i and length L_i (tokens in the cache after this step,
c_i < L_i, or c_i = L_i = 0 for a pad row).  Outputs: cu_seqlens_q,
cu_seqlens_k ([S+1]), context_lens (= L), slot_mapping (one entry per new
token, sequence by sequence) and the block tables packed to [S, max_blocks]
with -1 padding.
"""

from __future__ import annotations


def prepare_metadata(tables, num_cached, seq_lens, max_blocks: int, block_size: int = 256):
    S = len(seq_lens)
    cu_q = [0] * (S + 1)
    cu_k = [0] * (S + 1)
    slots = []
    packed = [[-1] * max_blocks for _ in range(S)]
    for i in range(S):
        c, L, tab = int(num_cached[i]), int(seq_lens[i]), list(tables[i])
        pad = c == 0 and L == 0
        if (not pad and not (0 <= c < L)) or len(tab) * block_size < L or len(tab) > max_blocks:
            raise ValueError(f"sequence {i}: need 0 <= cached < length <= blocks * block_size")
        cu_q[i + 1] = cu_q[i] + (L - c)
        cu_k[i + 1] = cu_k[i] + L
        for p in range(c, L):
            slots.append(tab[p // block_size] * block_size + p % block_size)
        packed[i][:len(tab)] = tab
    return {"cu_seqlens_q": cu_q, "cu_seqlens_k": cu_k, "context_lens": [int(x) for x in seq_lens],
            "slot_mapping": slots, "block_tables": packed}
