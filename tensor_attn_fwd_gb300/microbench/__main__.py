import json

from . import run

for rec in run():
    print(json.dumps(rec))
