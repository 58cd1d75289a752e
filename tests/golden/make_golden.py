"""Write tests/golden/oracle_digests.json: SHA-256 digests of the CPU
oracle's outputs on small seeded workloads.

Calls only the oracle and the seeded input generator.  Run it again (and say
why in the commit message) only when a reading of the pages changes the
oracle's arithmetic on purpose.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from oracle_pins import GOLDEN_CASES, _problem  # noqa: E402
from video_vae_decoder_qkv_gb300 import workloads as W  # noqa: E402


def main():
    out = {}
    for name, (spec, kw) in GOLDEN_CASES.items():
        inp = W.generate(spec)
        pb = _problem(spec, **kw)
        q, k, v, sc = oracle.prepare(pb, inp.qkv, inp.wq, inp.wk, inp.pos)
        h = hashlib.sha256()
        for t in (q, k, v):
            h.update(np.ascontiguousarray(t).tobytes())
        if sc is not None:
            h.update(np.asarray(sc, np.float32).tobytes())
        out[name] = h.hexdigest()
    path = os.path.join(HERE, "oracle_digests.json")
    with open(path, "w") as f:
        json.dump({"about": "SHA-256 of the oracle's q, k, v (and e4m3 descales) bytes; "
                            "written by tests/golden/make_golden.py", "digests": out}, f, indent=2)
        f.write("\n")
    print(path)


if __name__ == "__main__":
    main()
