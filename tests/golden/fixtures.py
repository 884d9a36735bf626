"""Reader for the key = value text fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def read(name):
    """Return {key: value-string} of a fixture, comments and blank lines skipped."""
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, value = line.partition("=")
            out[key.strip()] = value.strip()
    return out
