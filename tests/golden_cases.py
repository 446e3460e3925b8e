"""Reader for the text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def tree_geometry_cases():
    out = []
    with open(os.path.join(GOLDEN, "tree_geometry_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, mode, par, want = (c.strip() for c in line.split("|"))
            if par == "null":
                parent = None
            elif par == "":
                parent = []
            else:
                parent = [int(v) for v in par.split(",")]
            out.append((name, mode, parent, want))
    return out
