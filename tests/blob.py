"""Named views into a weight blob (test helper).

Tensor order of the loader in "bend-ml-llama 0.2.1.0, main.bend", section "Loading"
(t_layer): the embedding [V][d]; per layer ln1 [d], q [d][d], k [kvw][d], v [kvw][d],
o [d][d], ln2 [d], gate [f][d], up [f][d], down [d][f] (row = output); the final norm
[d]; for an untied head, lm_head [V][d].
"""
import numpy as np

LAYER_TENSORS = ("ln1", "q", "k", "v", "o", "ln2", "gate", "up", "down")


def layer_shapes(s):
    d, kvw, f = s.d, s.kvw, s.ffn
    return {"ln1": (d,), "q": (d, d), "k": (kvw, d), "v": (kvw, d), "o": (d, d),
            "ln2": (d,), "gate": (f, d), "up": (f, d), "down": (d, f)}


def views(shape, blob):
    """dict name -> view; layer tensors under (layer, name)."""
    out = {}
    o = 0

    def take(shp):
        nonlocal o
        n = int(np.prod(shp))
        v = blob[o:o + n].reshape(shp)
        o += n
        return v

    out["emb"] = take((shape.vocab, shape.d))
    ls = layer_shapes(shape)
    for i in range(shape.layers):
        for name in LAYER_TENSORS:
            out[(i, name)] = take(ls[name])
    out["lnf"] = take((shape.d,))
    if not shape.tied:
        out["lm_head"] = take((shape.vocab, shape.d))
    assert o == blob.size, (o, blob.size)
    return out
