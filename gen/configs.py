"""The five workloads of the tree-verification benchmark, with their sizes.

Each entry names the workload by what it is.  Shapes follow the Llama-3.1-8B target / EAGLE-3
draft head configuration printed in the qiita guide "EAGLE-3 and Medusa speculative decoding",
draft-head config (hidden 4096, 32 query heads, 8 KV heads, vocab 128256, draft vocab 32000),
and a 70B-shaped layer (64 query heads, hidden 8192) for the long-context case.
"""

CONFIGS = {
    1: dict(
        name="tiny-fp32-b1-l128-tree10-greedy",
        dtype="f32", B=1, prefix=("fixed", [128]), Hq=4, Hkv=1, d=64, Hd=256, V=2048,
        tree=("root3x2",), tokens=("rank", 0.7), rule="greedy", tau=0.0, eps=0.0, delta=0.0,
    ),
    2: dict(
        name="llama8b-b1-l2048-medusa63-typical",
        dtype="bf16", B=1, prefix=("fixed", [2048]), Hq=32, Hkv=8, d=128, Hd=4096, V=128256,
        tree=("static", (3, 3, 2, 2, 1), 63), tokens=("rank", 0.7), rule="typical",
        tau=1.0, eps=0.09, delta=0.3,
    ),
    3: dict(
        name="llama8b-b8-l512to8192-bfs127-rejection",
        dtype="bf16", B=8, prefix=("uniform", 512, 8192), Hq=32, Hkv=8, d=128, Hd=4096,
        V=128256, tree=("bfs", 127, 6), tokens=("iid", 0.7, 0.5), rule="rejection",
        tau=0.7, eps=0.0, delta=0.0,
    ),
    4: dict(
        name="eagle3-llama8b-b32-l4096-dynamic63-rejection",
        dtype="bf16", B=32, prefix=("fixed", [4096] * 32), Hq=32, Hkv=8, d=128, Hd=4096,
        V=128256, tree=("dynamic", 63, 8, 8), tokens=("dynamic", 32000, 0.5), rule="rejection",
        tau=1.0, eps=0.0, delta=0.0,
    ),
    5: dict(
        name="llama70b-b4-l32kto128k-bfs255-greedy",
        dtype="bf16", B=4, prefix=("fixed", [32768, 65536, 98304, 131072]), Hq=64, Hkv=8, d=128,
        Hd=8192, V=128256, tree=("bfs", 255, 8), tokens=("rank", 0.7), rule="greedy",
        tau=0.0, eps=0.0, delta=0.0,
    ),
}


def config_by_id(i):
    return dict(CONFIGS[i])
