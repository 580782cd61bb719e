"""Writes tests/golden/small_tile_stats.json: tile statistics of the Small
workload (8 frames of 16x24 patches, spatial frame window 2, temporal raster
window 40, 128x128 tiles), computed by the fp64 oracle alone.  A regression
pin: the values are the oracle's, produced by this script and nothing else."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

F, Hs, Ws, wf, ws = 8, 16, 24, 2, 40


def main():
    g = oracle.Geometry(F, Hs, Ws, wf=wf, ws=ws, bkv=128)
    out = {}
    for key, (kind, rounding) in {"spatial_exact": (oracle.SPATIAL, 0),
                                  "temporal_permuted_exact": (oracle.TEMPORAL_PERMUTED, 0),
                                  "temporal_fhw_exact": (oracle.TEMPORAL_FHW, 0),
                                  "spatial_rounded": (oracle.SPATIAL, 1),
                                  "temporal_permuted_rounded": (oracle.TEMPORAL_PERMUTED, 1)}.items():
        _, _, st = oracle.tile_map(kind, g, 128, 128, rounding)
        st.pop("ncols")
        out[key] = st
    with open(os.path.join(HERE, "small_tile_stats.json"), "w") as fh:
        json.dump(out, fh, indent=1, sort_keys=True)
        fh.write("\n")


if __name__ == "__main__":
    main()
