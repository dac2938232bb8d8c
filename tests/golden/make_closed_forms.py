"""Writes closed_forms.json: hand-derived exact results of tiny cases.

Each value is the closed form of its case, from the definitions on the pages
(cross-entropy: aprender-train wgpu_cross_entropy.rs, module doc and
``backward`` doc; top-k KL and top-k: cortiq-engine train_head.rs, module doc
and ``topk_rows`` doc).  The pages print no worked numbers.  This script uses
only the standard library: it calls neither the oracle nor the library.

    python tests/golden/make_closed_forms.py
"""
import json
import math
import os

G = {
    "_source": "Closed forms derived by hand from the definitions on the pages: "
               "aprender-train wgpu_cross_entropy.rs (module doc: loss = logsumexp(logits) - logits[label]; "
               "backward doc: grad = (softmax - one_hot) * scale) and cortiq-engine train_head.rs "
               "(module doc: L = sum_k p_T,k (log p_T,k - log p_S,id_k), dL/ds_j = p_S,j - p_T,j; "
               "topk_rows doc: probabilities renormalised over the k). Written by make_closed_forms.py.",
    "ce": [
        {"case": "two classes, logits [0, ln 3] give softmax [1/4, 3/4]; label 0",
         "logits": [0.0, math.log(3.0)], "label": 0, "scale": 1.0,
         "loss": math.log(4.0), "lse": math.log(4.0), "grad": [-0.75, 0.75]},
        {"case": "two classes, logits [0, ln 3]; label 1, scale 1/2",
         "logits": [0.0, math.log(3.0)], "label": 1, "scale": 0.5,
         "loss": math.log(4.0 / 3.0), "lse": math.log(4.0), "grad": [0.125, -0.125]},
        {"case": "uniform row of 1024 logits equal to 2.5: loss ln 1024, lse 2.5 + ln 1024",
         "logits_const": 2.5, "V": 1024, "label": 17, "scale": 0.25,
         "loss": math.log(1024.0), "lse": 2.5 + math.log(1024.0),
         "grad_label": 0.25 * (1.0 / 1024 - 1.0), "grad_other": 0.25 / 1024},
        {"case": "single-entry vocabulary: loss 0, gradient 0",
         "logits": [3.75], "label": 0, "scale": 1.0, "loss": 0.0, "lse": 3.75, "grad": [0.0]},
    ],
    "kl": [
        {"case": "uniform student over 4 columns, teacher support {1, 2} with probs 1/2 each: KL = ln 2",
         "logits": [0.0, 0.0, 0.0, 0.0], "tid": [1, 2], "tp": [0.5, 0.5], "coef": 1.0,
         "loss": math.log(2.0), "grad": [0.25, -0.25, -0.25, 0.25]},
        {"case": "student log-probs equal the teacher's on the support, -1e4 elsewhere: KL 0, gradient 0",
         "logits": [math.log(0.25), -1.0e4, math.log(0.75), -1.0e4], "tid": [2, 0], "tp": [0.75, 0.25],
         "coef": 2.0, "loss": 0.0, "grad": [0.0, 0.0, 0.0, 0.0]},
        {"case": "teacher mass on one id of a 2-column row with logits [0, ln 3]: KL = -ln(3/4)",
         "logits": [0.0, math.log(3.0)], "tid": [1], "tp": [1.0], "coef": 0.5,
         "loss": -math.log(0.75), "grad": [0.125, -0.125]},
    ],
    "topk": [
        {"case": "ties go to the lower column and -0.0 equals +0.0",
         "logits": [3.0, 1.0, 3.0, 2.0, -0.0, 0.0, 1.0], "k": 6,
         "ids": [0, 2, 3, 1, 6, 4],
         "probs_unnormalised": [1.0, 1.0, math.exp(-1.0), math.exp(-2.0), math.exp(-2.0), math.exp(-3.0)]},
        {"case": "k = 1 is the first maximum, probability 1",
         "logits": [-1.0, 5.0, 5.0, 4.0], "k": 1, "ids": [1], "probs_unnormalised": [1.0]},
    ],
    "memory_figure": {
        "case": "only [seq] log-sum-exp values are kept instead of the [seq x vocab] fp32 softmax; "
                "for vocab 32000 and seq 512 the saving is quoted as about 62 MB",
        "seq": 512, "vocab": 32000, "bytes": 65536000, "mib": 62.5,
    },
}

if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "closed_forms.json"), "w") as f:
        json.dump(G, f, indent=1)
