"""Plain fp64 CPU oracle for tree verification in Medusa/EAGLE-style speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never calls it, and it shares no
code with the CUDA library (no common kernels, headers, helpers, tables or constant
generators).  Both sides read the same seeded inputs from ``gen/``.

Pages this oracle follows (cited by short tag in every module):

* [MTP]   tech-tldr.com, "多トークン予測（Medusa・EAGLE）" (multi-token prediction).
* [GLOSS] jisaku.com glossary, "Medusa（マルチヘッド投機的デコーディング）".
* [GUIDE] qiita.com, "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド".

Pins (see tests/test_oracle_*.py): the ancestor mask against a graph library's ancestor sets and
the tree figure of [GUIDE] section "Tree Attention"; attention against a library causal
attention for single-chain trees and against plain decoding for a single node; row statistics
against closed forms and library routines; path selection against the invariants of [GUIDE]
section "棄却サンプリング" and [MTP] section "ツリー検証"; rejection sampling against the target
distribution by a chi-square test over 10^6 seeded trials (with a planted-mistake negative
control); the margin detector (greedy gap, typical log-ratio, rejection ratio band, bonus
window) and the draft-to-target scatter against hand-computed cases; Philox against an
independent library implementation; Medusa expansion against the
18-path example of [GLOSS] section "ツリー構造の候補構築", brute-force top-k and the input
generator's independent topology builder.  Nothing is "parity unpinned".
"""

from .philox import philox4x32_10, uniforms  # noqa: F401
from .tree import (validate_tree, ancestors_or_self, depths, tree_mask, root_to_leaf_paths,  # noqa: F401
                   children)
from .attention import tree_attention, tree_attention_rows  # noqa: F401
from .lmhead import logits, row_stats  # noqa: F401
from .accept import verify_request, verify_accept, draft_in_target_vocab, MARGIN  # noqa: F401
from .compact import compact_kv  # noqa: F401
from .medusa import head_topk, cartesian_tuples, pruned_topology, medusa_expand  # noqa: F401
from .paged import gather_paged, scatter_paged  # noqa: F401
from .eagle import expand_layer, select_tree  # noqa: F401
