"""Plain restatement of GraniKV's per-step backend rule.  TEST INFRASTRUCTURE ONLY.

"3 GraniKV", per-step dispatch, and "B.4 Per-Step Dispatch Trace": each decode step computes
the effective GEMM height M_eff = B * n_q / n_kv of the realised batch and runs the dense
(batched-GEMM) prefix backend when M_eff >= M_sat, else the cascade backend.  Under several
distinct prefixes the pages batch each prefix against its own slab ("B.8 Multi-prefix
sensitivity": class-local dense batching), so the rule is applied per prefix group with B the
number of requests sharing that slab.  Requests whose prefix is not in HOT form no group.
"""

from __future__ import annotations

from typing import Dict, List, Sequence

DENSE = "dense"
CASCADE = "cascade"


def m_eff(batch_size: int, n_q: int, n_kv: int) -> int:
    return batch_size * n_q // n_kv


def plan_groups(slab_ids: Sequence[int], n_q: int, n_kv: int, m_sat: int) -> List[Dict]:
    """Groups in order of first appearance of each slab id; members in request order."""
    order: List[int] = []
    members: Dict[int, List[int]] = {}
    for b, sid in enumerate(slab_ids):
        if sid < 0:
            continue
        if sid not in members:
            members[sid] = []
            order.append(sid)
        members[sid].append(b)
    out = []
    for sid in order:
        me = m_eff(len(members[sid]), n_q, n_kv)
        out.append({"slab": sid, "requests": members[sid], "m_eff": me,
                    "backend": DENSE if me >= m_sat else CASCADE})
    return out
