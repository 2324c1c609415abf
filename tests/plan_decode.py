"""Test helper: decode the binary plan layout documented in
sm_load_balancing_gb300/csrc/plan_layout.h into per-CTA segment lists."""
import numpy as np

PH_WORDS = 16
MAGIC = 0x534B4431


def _align4(x):
    return (x + 3) & ~3


def offsets(batch, hkv, n):
    items = batch * hkv
    cap = items + n
    cta_off = PH_WORDS
    segs = cta_off + _align4(n + 1)
    nsplit = segs + 4 * cap
    slot0 = nsplit + items
    return dict(cta_off=cta_off, segs=segs, nsplit=nsplit, slot0=slot0, words=slot0 + items)


def decode(plan):
    w = np.asarray(plan, dtype=np.int32)
    assert w[0] == MAGIC
    batch, hkv, n = int(w[1]), int(w[2]), int(w[3])
    o = offsets(batch, hkv, n)
    nseg = int(w[6])
    cta_off = w[o["cta_off"]:o["cta_off"] + n + 1]
    segs = w[o["segs"]:o["segs"] + 4 * nseg].reshape(-1, 4)
    per_cta = []
    for c in range(n):
        per_cta.append([tuple(int(x) for x in segs[k]) for k in range(cta_off[c], cta_off[c + 1])])
    items = batch * hkv
    return dict(batch=batch, hkv=hkv, n=n, granule=int(w[4]), nitems=int(w[5]), nseg=nseg,
                nslots=int(w[7]), total=int(w[8]), mode=int(w[9]), cap=int(w[10]), err=int(w[11]),
                segments=per_cta, nsplit=w[o["nsplit"]:o["nsplit"] + items].tolist(),
                slot0=w[o["slot0"]:o["slot0"] + items].tolist())
