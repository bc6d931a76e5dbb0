"""Writes the two hand-derived fixtures in this folder.

Nothing here calls the oracle or the CUDA path: the numbers are the closed-form
results of the derivation recorded in each file (two keys, scores 0 and ln 3,
so the softmax row is exactly [1/4, 3/4]; a second query with equal scores,
[1/2, 1/2]; a masked variant where only key 0 is attended), and a small integer
example of the Ulysses index map.  Run from the repository root:
``python tests/golden/make_golden.py``.
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def attention_doc():
    ln3 = math.log(3.0)
    doc = {
        "source": "Hand-derived closed form (no page prints a worked example). Softmax attention as "
                  "defined for the SDPA forward/backward op pair in 'Fix double transpose of K/V in "
                  "templated attention backward' (description and Test paragraphs) and the "
                  "bool-mask-to-additive-bias reading of its follow-up item 2.",
        "derivation": [
            "B=1,S=2,H=1,D=2. k0=[0,0], k1=[c*ln3, c*5] with c=1/scale, so scale*q0.k1 = ln3 for q0=[1,0]. "
            "v0=[1,0], v1=[3,2]. q1=[0,0].",
            "query 0: s=[0, ln3] -> P=[1/4, 3/4], LSE=ln4, O=[1/4+9/4, 6/4]=[2.5, 1.5]",
            "query 1: s=[0, 0]   -> P=[1/2, 1/2], LSE=ln2, O=[2, 1]",
            "dO0=[1,0], dO1=[0,1]; dP0=[1,3], Delta0=2.5; dP1=[0,2], Delta1=1",
            "dS0=[1/4(1-2.5), 3/4(3-2.5)]=[-0.375, 0.375]; dS1=[-0.5, 0.5]",
            "dQ_i = scale*sum_j dS_ij k_j ; dK_j = scale*sum_i dS_ij q_i ; dV_j = sum_i P_ij dO_i",
            "masked case (key 1 False): every row attends key 0 only: P=[1,0], LSE=0, O=v0, dS=0, "
            "dQ=dK=0, dV0=dO0+dO1, dV1=0",
        ],
        "cases": [],
    }
    for scale in (1.0, 0.5):
        c = 1.0 / scale
        q = [[[[1.0, 0.0]], [[0.0, 0.0]]]]
        k = [[[[0.0, 0.0]], [[c * ln3, c * 5.0]]]]
        v = [[[[1.0, 0.0]], [[3.0, 2.0]]]]
        do = [[[[1.0, 0.0]], [[0.0, 1.0]]]]
        ds = [[-0.375, 0.375], [-0.5, 0.5]]
        kk = [[0.0, 0.0], [c * ln3, c * 5.0]]
        qq = [[1.0, 0.0], [0.0, 0.0]]
        dq = [[scale * sum(ds[i][j] * kk[j][d] for j in range(2)) for d in range(2)] for i in range(2)]
        dk = [[scale * sum(ds[i][j] * qq[i][d] for i in range(2)) for d in range(2)] for j in range(2)]
        doc["cases"].append({
            "name": f"two_keys_scale_{scale}", "scale": scale, "mask": None,
            "q": q, "k": k, "v": v, "do": do,
            "o": [[[[2.5, 1.5]], [[2.0, 1.0]]]],
            "lse": [[[math.log(4.0), math.log(2.0)]]],
            "dq": [[[dq[0]], [dq[1]]]],
            "dk": [[[dk[0]], [dk[1]]]],
            "dv": [[[[0.25, 0.5]], [[0.75, 0.5]]]],
        })
        doc["cases"].append({
            "name": f"two_keys_masked_scale_{scale}", "scale": scale, "mask": [[1, 0]],
            "q": q, "k": k, "v": v, "do": do,
            "o": [[[[1.0, 0.0]], [[1.0, 0.0]]]],
            "lse": [[[0.0, 0.0]]],
            "dq": [[[[0.0, 0.0]], [[0.0, 0.0]]]],
            "dk": [[[[0.0, 0.0]], [[0.0, 0.0]]]],
            "dv": [[[[1.0, 1.0]], [[0.0, 0.0]]]],
        })
    return doc


def relayout_doc():
    return {
        "source": "Hand-written index example of the Ulysses exchange ('[attention] Add Ulysses Anything "
                  "backward', What does this PR do: all-to-all with separate partition metadata; trim each "
                  "gathered mask shard before concatenation).",
        "P": 2, "shard_lens": [3, 1], "cap": 3, "B": 1, "H": 2, "D": 1,
        "x_shards_note": "x[p][b][s][h][d]; value = 100*p + 10*s + h; shard 1 rows 1,2 are padding (0)",
        "x_shards": [[[[[0], [1]], [[10], [11]], [[20], [21]]]],
                     [[[[100], [101]], [[0], [0]], [[0], [0]]]]],
        "y_groups_note": "y[g][b][n][h'][d]: group g holds head g of rows (shard0 rows 0..2, shard1 row 0)",
        "y_groups": [[[[[0]], [[10]], [[20]], [[100]]]], [[[[1]], [[11]], [[21]], [[101]]]]],
        "mask_gathered": [[[1, 1, 0]], [[1, 0, 0]]],
        "mask_assembled": [[1, 1, 0, 1]],
        "mask_untrimmed_defect": [[1, 1, 0, 1, 0, 0]],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "attention_two_keys.json"), "w") as f:
        json.dump(attention_doc(), f, indent=1)
    with open(os.path.join(HERE, "ulysses_relayout_small.json"), "w") as f:
        json.dump(relayout_doc(), f, indent=1)
