"""Reader of the pipe-separated text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append([c.strip() for c in line.split("|")])
    return out


def parse_shapes(text):
    return [tuple(int(x) for x in s.split(",")) for s in text.split(";")]
