"""Reader for the golden fixture files: '# ...' header lines, then rows of
'<i> <j> <value> <value> ...'."""


def load_fixture(path):
    rows = {}
    with open(path) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = line.split()
            rows[(int(p[0]), int(p[1]))] = [float(x) for x in p[2:]]
    return rows
