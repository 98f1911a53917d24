"""Writes worked_examples.json: hand-derived closed forms of tiny attention problems.

The pages print no numeric example, so each value below is a closed form derived by hand
from the pages' equations and evaluated here with the standard library only. It calls
neither the oracle nor the CUDA path. Inputs are small integers, which are exact in bf16.
Run: python tests/golden/make_worked_examples.py
"""
import json
import math
import os

E = math.e

GOLD = {
    "_about": "Hand-derived worked examples for the split-KV decode oracle. The pages print no "
              "numeric example; each value is the closed form in 'expr', evaluated in double "
              "precision by make_worked_examples.py. Inputs are small integers (exact in bf16).",
    "two_token": {
        "cite": "Infinite-LLM notes, section 分布式注意力机制的通信挑战 (full attention with the "
                "global max m_g) and the MicroAttention / aggregation equations "
                "(DistAttention 的等价数学变换, 结果聚合与通信开销降低)",
        "d": 2, "scale": 1.0, "q": [1, 0], "K": [[0, 0], [1, 0]], "V": [[1, 0], [0, 1]],
        "expr": "logits (0, 1); out = (1/(1+e), e/(1+e)); m = 1; e_g = 1 + exp(-1)",
        "out": [1 / (1 + E), E / (1 + E)], "m": 1.0, "e": 1 + math.exp(-1),
        "partials_expr": "chunk {k1}: (m=0, e=1, MA=v1); chunk {k2}: (m=1, e=1, MA=v2)",
        "partials": [[0.0, 1.0, [1, 0]], [1.0, 1.0, [0, 1]]],
    },
    "three_token": {
        "cite": "Infinite-LLM notes, full attention and MicroAttention / aggregation equations",
        "d": 1, "scale": 1.0, "q": [1], "K": [[0], [1], [2]], "V": [[1], [2], [3]],
        "expr": "logits (0, 1, 2); out = (1 + 2e + 3e^2)/(1 + e + e^2); m = 2; "
                "e_g = 1 + exp(-1) + exp(-2)",
        "out": [(1 + 2 * E + 3 * E * E) / (1 + E + E * E)], "m": 2.0,
        "e": 1 + math.exp(-1) + math.exp(-2),
    },
    "three_token_half_scale": {
        "cite": "Infinite-LLM notes, full attention equations, with a scale factor of 0.5 "
                "applied to the logits",
        "d": 1, "scale": 0.5, "q": [1], "K": [[0], [1], [2]], "V": [[1], [2], [3]],
        "expr": "logits (0, 0.5, 1); out = (1 + 2e^0.5 + 3e)/(1 + e^0.5 + e); m = 1; "
                "e_g = exp(-1) + exp(-0.5) + 1",
        "out": [(1 + 2 * math.exp(0.5) + 3 * E) / (1 + math.exp(0.5) + E)], "m": 1.0,
        "e": math.exp(-1) + math.exp(-0.5) + 1,
    },
    "page_score": {
        "cite": "LServe article §3.1.2 (动态稀疏的层次化选择): per-channel k_max/k_min and a "
                "query-vs-statistics page score, read as sum_d max(q_d kmax_d, q_d kmin_d)",
        "q": [1, -2], "keys": [[3, -4], [-1, 1], [2, 0]],
        "expr": "kmax = (3, 1), kmin = (-1, -4); score = max(3, -1) + max(-2, 8) = 11; "
                "q.k = (11, -3, 2)",
        "kmax": [3, 1], "kmin": [-1, -4], "score": 11.0, "qk": [11.0, -3.0, 2.0],
    },
    "topk": {
        "cite": "LServe article §3.1.2 (keep the K highest-scoring physical pages); ties go to "
                "the lower page index; output ascending, -1 padded",
        "scores": [5, 7, 7, 1, 9],
        "cases": [[3, [1, 2, 4]], [2, [1, 4]], [1, [4]], [7, [0, 1, 2, 3, 4, -1, -1]]],
    },
    "streaming_rows": {
        "cite": "LServe article §3.1.1 (流式头: attention sinks plus a local window); decode "
                "has no future tokens, so the window is the last `local` tokens",
        "sinks": 4, "local": 8,
        "cases": [[20, [0, 1, 2, 3, 12, 13, 14, 15, 16, 17, 18, 19]],
                  [12, list(range(12))], [10, list(range(10))], [3, [0, 1, 2]], [0, []]],
    },
}

if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_examples.json")
    with open(path, "w") as f:
        json.dump(GOLD, f, indent=1, ensure_ascii=False)
        f.write("\n")
    print("wrote", path)
